// Device code of gbtopk: batched variable-length exact top-K on sm_103a.
//
// Every call's launch geometry depends only on (rows, width, top_k, dtype),
// never on the seq_lens / lengths contents, so any call can be captured in a
// CUDA graph and replayed with new lengths (TensorRT-LLM PR #17821, the
// run_varlen commits).  Per row (valid length n, from the FlashInfer
// `top_k_varlen` seq_lens formula or from the page-table calls' lengths and
// row_starts):
//   * n == 0 or n <= k -> every valid column, then -1 (short path);
//   * widths up to 2048 without the sorted order: one warp per row, a
//     warp-private radix select (small16_kernel for 16-bit rows: the row
//     staged by one bulk copy and turned into packed pair keys in place;
//     small_kernel for fp32: keys in registers);
//   * rows of up to 64 KB: one block per row (row_kernel): the
//     row is staged in shared memory by one bulk copy, a threshold is
//     guessed from a strided sample, the elements at or above it are kept
//     and selected exactly in shared memory;
//   * longer rows (split plans), top_k <= 2048 and batches of at most 2048
//     (row, 64 KB chunk) slots: row_kernel makes each row's guess (the
//     self-sampling guess of TensorRT-LLM PR #17821, its key range widened
//     to the hint's argmax), then chunk_kernel runs one block per chunk:
//     the chunk is filtered against the guess into a candidate segment and
//     the row's last block (atomic ticket) selects the row in its own
//     shared memory (finalize_row);
//   * other split plans: row_kernel's guesses, then the persistent
//     stream_kernel filters every 64 KB chunk through a bulk-copy ring of
//     three stages, then final_kernel selects each row (finalize_row).
// The three launches of a call are chained by programmatic dependent launch.
// A guess that was too high, a candidate segment that overflowed or a
// bounded wait that gave up sends the row through an exact radix select
// over global memory (count-crossing check), so the result never depends on
// the guess.  Ranking uses order-preserving integer keys (signed zeros
// equal; +-inf and denormals exact), so no float compare depends on
// flush-to-zero.
#include <cstddef>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gbtopk_internal.h"

namespace gbtopk {

// Trace rows of each kernel's blocks (GBTOPK_TRACE builds): row kernel from 0,
// stream kernel from kTraceStream, finalize kernel from kTraceFinal.
constexpr int kTraceStream = 32768;
constexpr int kTraceFinal = 40960;
constexpr int kTraceChunk = 8192;  // chunk kernel blocks (up to 24576 of them)

#ifdef GBTOPK_TRACE
// Phase stamps of the first kTraceBlocks blocks, for builds compiled with
// -DGBTOPK_TRACE (read back by gbtopk_trace_read): SM cycles (%clock64),
// cheap to read.  Each block also leaves one anchor at its end, slot 30 =
// %clock64 and slot 31 = %globaltimer (ns) read together, which places its
// cycle stamps on the common time axis.  A %globaltimer read slows the
// warp that makes it for thousands of cycles afterwards, so it is taken
// once per block, after the traced work.
constexpr int kTraceBlocks = 1 << 16;
__device__ unsigned long long g_trace[kTraceBlocks][32];
// Each kernel declares kTraceBase: its blocks use g_trace[kTraceBase + block].
#define GBTOPK_TRACE_POINT(slot, value)                                                      \
    do {                                                                                     \
        if (threadIdx.x == 0 && kTraceBase + blockIdx.x < kTraceBlocks) {                    \
            unsigned long long t_;                                                           \
            asm volatile("mov.u64 %0, %%clock64;" : "=l"(t_));                               \
            g_trace[kTraceBase + blockIdx.x][slot] = ((slot) == 7 || (slot) == 15) ? (value) : t_; \
        }                                                                                    \
    } while (0)
// g_trace[index][slot] = the current cycle count (value < 0) or value, from any thread.
#define GBTOPK_TRACE_SET(index, slot, value)                                              \
    do {                                                                                 \
        if ((index) < kTraceBlocks) {                                                    \
            long long v_ = (value);                                                      \
            if (v_ < 0) asm volatile("mov.u64 %0, %%clock64;" : "=l"(v_));              \
            g_trace[(index)][(slot)] = static_cast<unsigned long long>(v_);              \
        }                                                                                \
    } while (0)
// The block's anchor (thread 0, at the end of the block's traced work).
#define GBTOPK_TRACE_ANCHOR()                                                                \
    do {                                                                                     \
        if (threadIdx.x == 0 && kTraceBase + blockIdx.x < kTraceBlocks) {                    \
            unsigned long long c_, g_;                                                       \
            asm volatile("mov.u64 %0, %%clock64;\n\tmov.u64 %1, %%globaltimer;" : "=l"(c_), "=l"(g_)); \
            g_trace[kTraceBase + blockIdx.x][30] = c_;                                       \
            g_trace[kTraceBase + blockIdx.x][31] = g_;                                       \
        }                                                                                    \
    } while (0)
#else
#define GBTOPK_TRACE_POINT(slot, value) \
    do {                                \
    } while (0)
#define GBTOPK_TRACE_SET(index, slot, value) \
    do {                                     \
    } while (0)
#define GBTOPK_TRACE_ANCHOR() \
    do {                      \
    } while (0)
#endif

namespace {

// ---------------------------------------------------------------- keys

template <int DT>
struct Elem;

template <>
struct Elem<0> {  // fp32
    using raw_t = uint32_t;
    static constexpr int kBytes = 4;
    static constexpr int kKeyBits = 32;
    static constexpr uint32_t kLowest = 0xFF7FFFFFu;   // -FLT_MAX
    __device__ __forceinline__ static uint32_t key(uint32_t u) {
        u = (u == 0x80000000u) ? 0u : u;
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
};

struct Elem16 {
    using raw_t = uint16_t;
    static constexpr int kBytes = 2;
    static constexpr int kKeyBits = 16;
    __device__ __forceinline__ static uint32_t key(uint32_t u) {
        u &= 0xFFFFu;
        u = (u == 0x8000u) ? 0u : u;
        return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
    }
};

template <>
struct Elem<1> : Elem16 {  // bf16
    static constexpr uint32_t kLowest = 0xFF7Fu;
};

template <>
struct Elem<2> : Elem16 {  // fp16
    static constexpr uint32_t kLowest = 0xFBFFu;
};

// ---------------------------------------------------------------- control block

struct Ctrl {
    unsigned long long bar;  // mbarrier for the bulk copy
    uint32_t bcast[8];
    uint32_t sel_count;
    uint32_t tie_count;
    uint32_t cand_count;
    uint32_t b_count;
    uint32_t key_max;
    uint32_t abort_flag;     // stream kernel: a bounded wait gave up, stop streaming
    uint32_t pad[2];
    uint32_t scan[72];
    alignas(16) uint32_t rhist[256];  // radix-select digit histogram (read with vector loads)
    uint32_t key_min;
    unsigned long long full[kStages];   // stream ring: stage filled (bulk copy landed)
    unsigned long long empty[kStages];  // stream ring: stage read by every consumer warp
    // stream ring: per stage and parity, candidates reserved (low word) and
    // consumer warps done (high word) for the stage's chunk
    unsigned long long scombo[2][kStages];
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");
static_assert(offsetof(Ctrl, rhist) % 16 == 0, "vector loads of the digit histogram");

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte permute (PTX prmt, generic mode): selector nibble i picks, for result byte i,
// one of the bytes 0-7 of {b, a}; a nibble with bit 3 set replicates that byte's
// sign bit over the result byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Claims consecutive slots of a shared counter for the lanes with `pred`
// (one atomic per warp).  Every lane of the warp must call it.
__device__ __forceinline__ uint32_t warp_claim(uint32_t *counter, bool pred) {
    const uint32_t m = __ballot_sync(0xffffffffu, pred);
    uint32_t base = 0;
    if (m) {
        const int leader = __ffs(m) - 1;
        if (static_cast<int>(lane_id()) == leader) base = atomicAdd(counter, __popc(m));
        base = __shfl_sync(0xffffffffu, base, leader);
    }
    return base + __popc(m & lanemask_lt());
}

// Histogram increment aggregated over lanes that hit the same bin.
__device__ __forceinline__ void warp_hist_add(uint32_t *hist, uint32_t bin, bool pred) {
    const uint32_t m = __ballot_sync(0xffffffffu, pred);
    if (pred) {
        const uint32_t peers = __match_any_sync(m, bin);
        if (static_cast<int>(lane_id()) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
}

// Inclusive prefix sum over the lanes of a full warp.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= static_cast<uint32_t>(off)) v += y;
    }
    return v;
}

// Exclusive prefix sum of one value per thread (thread order).  All threads.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Ctrl &c, uint32_t &total) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= static_cast<uint32_t>(off)) incl += y;
    }
    if (lane == 31) c.scan[warp] = incl;
    __syncthreads();
    if (threadIdx.x < 32) {
        const uint32_t w = lane < nw ? c.scan[lane] : 0u;
        uint32_t s = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= static_cast<uint32_t>(off)) s += y;
        }
        c.scan[32 + lane] = s - w;
        if (lane == 31) c.scan[64] = s;
    }
    __syncthreads();
    total = c.scan[64];
    const uint32_t r = c.scan[32 + warp] + incl - v;
    __syncthreads();
    return r;
}

// Block-wide min and max of one key per thread into c.key_min / c.key_max
// (which thread 0 must have reset to ~0u / 0 before a preceding barrier).
__device__ __forceinline__ void block_minmax(uint32_t kmin, uint32_t kmax, Ctrl &c) {
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane_id() == 0) {
        atomicMin(&c.key_min, kmin);
        atomicMax(&c.key_max, kmax);
    }
    __syncthreads();
}

// Counts from the top over NB counters: calls f(b, above, cnt) once for every
// bin b, with above = the sum of the counts of the bins > b.  Thread t owns
// the run of NB / NT bins that follows thread t - 1's from the top and reads
// it with vector loads (at most 2-way bank conflicts); one block scan of the
// runs' sums gives each run its start.  Ends with a barrier (the counters
// may be rewritten by f; c.scan is free again).
template <int NT, int NB, class F>
__device__ __forceinline__ void scan_from_top(const uint32_t *hist, Ctrl &c, F f) {
    constexpr int BPT = NB / NT;
    static_assert(BPT * NT == NB && (BPT == 2 || BPT % 4 == 0), "bins per thread");
    const int lo = NB - BPT * (static_cast<int>(threadIdx.x) + 1);  // lowest bin of the run
    uint32_t cnt[BPT];
    if constexpr (BPT == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(hist + lo);
        cnt[0] = v.x;
        cnt[1] = v.y;
    } else {
#pragma unroll
        for (int q = 0; q < BPT / 4; ++q) {
            const uint4 v = *reinterpret_cast<const uint4 *>(hist + lo + 4 * q);
            cnt[4 * q] = v.x;
            cnt[4 * q + 1] = v.y;
            cnt[4 * q + 2] = v.z;
            cnt[4 * q + 3] = v.w;
        }
    }
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) sum += cnt[j];
    uint32_t tot;
    uint32_t above = block_excl_scan(sum, c, tot);
#pragma unroll
    for (int j = BPT - 1; j >= 0; --j) {
        f(static_cast<uint32_t>(lo + j), above, cnt[j]);
        above += cnt[j];
    }
    __syncthreads();
}

// ---------------------------------------------------------------- bulk copy (TMA)

__device__ __forceinline__ void mbar_init(unsigned long long *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                          unsigned long long *bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try(unsigned long long *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of the barrier; gives up after `limit` polls.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity, uint32_t limit = kSpinLimit) {
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try(bar, parity)) return true;
    return false;
}

// mbar_wait that also gives up when *abort becomes nonzero (checked every
// 64 polls): 1 when the phase completed, 0 on the poll limit, 2 on abort.
__device__ __forceinline__ int mbar_wait_or_abort(unsigned long long *bar, uint32_t parity, uint32_t limit,
                                                  const volatile uint32_t *abort) {
    for (uint32_t it = 0; it < limit; ++it) {
        if (mbar_try(bar, parity)) return 1;
        if ((it & 63u) == 63u && *abort) return 2;
    }
    return 0;
}

template <typename R>
__device__ __forceinline__ uint32_t ldg_raw(const R *p) {
    return static_cast<uint32_t>(__ldg(p));
}

// ---------------------------------------------------------------- key sources
// A source yields (key, column index, raw bits) for item i.  kBatch items
// per thread are fetched before any is used, so global-memory sources keep
// several loads in flight per thread.

template <int DT>
struct StageSrc {  // a row (or chunk) staged in shared memory
    static constexpr int kBatch = 4;
    const typename Elem<DT>::raw_t *s;
    __device__ __forceinline__ void get(int64_t i, uint32_t &key, uint32_t &idx, uint32_t &raw) const {
        raw = s[i];
        key = Elem<DT>::key(raw);
        idx = static_cast<uint32_t>(i);
    }
};

template <int DT>
struct GlobalSrc {  // a row read straight from global memory
    static constexpr int kBatch = 8;
    const typename Elem<DT>::raw_t *g;
    __device__ __forceinline__ void get(int64_t i, uint32_t &key, uint32_t &idx, uint32_t &raw) const {
        raw = ldg_raw(g + i);
        key = Elem<DT>::key(raw);
        idx = static_cast<uint32_t>(i);
    }
};

template <int DT>
struct PairSrc {  // (raw, column) pairs in shared memory
    static constexpr int kBatch = 4;
    const uint2 *p;
    __device__ __forceinline__ void get(int64_t i, uint32_t &key, uint32_t &idx, uint32_t &raw) const {
        const uint2 v = p[i];
        raw = v.x;
        key = Elem<DT>::key(v.x);
        idx = v.y;
    }
};

// Visits items [0, cnt) of a source, kBatch per thread per pass, calling
// f(valid, key, idx, raw) for each.  Every thread makes the same number of
// calls (warp-collective operations inside f are allowed).
template <class S, class F>
__device__ __forceinline__ void for_each_item(const S &s, int64_t cnt, F &&f) {
    constexpr int B = S::kBatch;
    const int64_t step = static_cast<int64_t>(blockDim.x) * B;
    for (int64_t base = 0; base < cnt; base += step) {
        uint32_t key[B], idx[B], raw[B];
        bool valid[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * blockDim.x + threadIdx.x;
            valid[u] = i < cnt;
            key[u] = idx[u] = raw[u] = 0;
            if (valid[u]) s.get(i, key[u], idx[u], raw[u]);
        }
#pragma unroll
        for (int u = 0; u < B; ++u) f(valid[u], key[u], idx[u], raw[u]);
    }
}

// Ranking modes for block_select: by key, or (deterministic ties) among the
// items whose key equals t, smallest column first.
struct RankByKey {
    __device__ __forceinline__ bool operator()(uint32_t key, uint32_t, uint32_t &k) const {
        k = key;
        return true;
    }
};

// Tie modes (among values equal to the k-th): 0 any, 1 the smallest
// columns, 2 the largest.  tie_key orders the preferred columns first.
__device__ __forceinline__ uint32_t tie_key(uint32_t col, int tie) { return tie == 2 ? ~col : col; }

struct RankTieColumn {
    uint32_t t;
    int tie;
    __device__ __forceinline__ bool operator()(uint32_t key, uint32_t idx, uint32_t &k) const {
        k = ~tie_key(idx, tie);
        return key == t;
    }
};

// Block-wide radix select: the r-th largest (1-based) ranked value among the
// items of `src` admitted by `mode`, digit by digit from the top (8-bit
// digits, 256-bin shared histogram, warp-aggregated increments).  With
// ROUNDS < KEY_BITS/8 the result is the r-th largest value truncated to its
// top 8*ROUNDS bits (a lower bound of it).  Returns the value and, in `gt`,
// how many admitted items rank strictly above it (exact when every digit
// was resolved).  Requires 1 <= r <= number of admitted items.
template <int KEY_BITS, int ROUNDS, class Src, class Mode>
__device__ void block_select(const Src &src, const Mode &mode, int64_t cnt, uint32_t r,
                             uint32_t *hist, Ctrl &c, uint32_t &out_key, uint32_t &out_gt) {
    uint32_t prefix = 0, mask = 0, rem = r;
#pragma unroll 1
    for (int round = 0; round < ROUNDS; ++round) {
        const int shift = KEY_BITS - 8 * (round + 1);
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for_each_item(src, cnt, [&](bool valid, uint32_t key, uint32_t idx, uint32_t) {
            uint32_t k = 0;
            const bool ok = valid && mode(key, idx, k) && (k & mask) == prefix;
            warp_hist_add(hist, (k >> shift) & 255u, ok);
        });
        __syncthreads();
        if (threadIdx.x < 32) {
            const uint32_t lane = lane_id();
            uint32_t cnts[8], s = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cnts[j] = hist[255 - 8 * lane - j];
                s += cnts[j];
            }
            uint32_t incl = s;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= static_cast<uint32_t>(off)) incl += y;
            }
            const uint32_t excl = incl - s;
            const bool has = excl < rem && rem <= incl;
            const uint32_t bal = __ballot_sync(0xffffffffu, has);
            if (bal == 0u) {
                if (lane == 0) {  // unreachable when 1 <= r <= count
                    c.bcast[0] = 0;
                    c.bcast[1] = 0;
                }
            } else if (static_cast<int>(lane) == __ffs(bal) - 1) {
                uint32_t acc = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (acc + cnts[j] >= rem) {
                        c.bcast[0] = 255u - 8u * lane - static_cast<uint32_t>(j);
                        c.bcast[1] = acc;
                        break;
                    }
                    acc += cnts[j];
                }
            }
        }
        __syncthreads();
        prefix |= c.bcast[0] << shift;
        mask |= 0xFFu << shift;
        rem -= c.bcast[1];
        __syncthreads();
    }
    out_key = prefix;
    out_gt = r - rem;
}

// Writes every item with key > t into sel[base + 0 ..) and `need_ties`
// items with key == t into sel[base + gt ..).  With a tie mode it keeps the
// ties whose tie_key is <= tie_col_max (exactly need_ties of them).
template <int DT, class S>
__device__ void collect(const S &s, int64_t cnt, uint32_t t, uint32_t gt, uint32_t need_ties,
                        int tie, uint32_t tie_col_max, uint2 *sel, uint32_t base, Ctrl &c) {
    if (threadIdx.x == 0) {
        c.sel_count = 0;
        c.tie_count = 0;
    }
    __syncthreads();
    for_each_item(s, cnt, [&](bool valid, uint32_t key, uint32_t idx, uint32_t raw) {
        const bool above = valid && key > t;
        const bool keep = valid && key == t && (!tie || tie_key(idx, tie) <= tie_col_max);
        const uint32_t slot = warp_claim(&c.sel_count, above);
        if (above) sel[base + slot] = make_uint2(raw, idx);
        const uint32_t tslot = warp_claim(&c.tie_count, keep);
        if (keep && tslot < need_ties) sel[base + gt + tslot] = make_uint2(raw, idx);
    });
    __syncthreads();
}

// Exact top-k (n > k) of a source into sel[0..k).
template <int DT, class S>
__device__ void exact_select(const S &s, int64_t n, int k, int tie, uint2 *sel, uint32_t *hist,
                             Ctrl &c) {
    constexpr int KB = Elem<DT>::kKeyBits;
    uint32_t t, gt;
    block_select<KB, KB / 8>(s, RankByKey{}, n, static_cast<uint32_t>(k), hist, c, t, gt);
    const uint32_t need_ties = static_cast<uint32_t>(k) - gt;
    uint32_t col_max = 0xFFFFFFFFu;
    if (tie) {
        uint32_t kk, g2;
        block_select<32, 4>(s, RankTieColumn{t, tie}, n, need_ties, hist, c, kk, g2);
        col_max = ~kk;
    }
    collect<DT>(s, n, t, gt, need_ties, tie, col_max, sel, 0, c);
}

// ---------------------------------------------------------------- row geometry and output

// Request b of a score row when rows are grouped by cu_seqlens_q
// (cu_seqlens_q[b] <= row < cu_seqlens_q[b + 1]), or -1 when none covers it.
__device__ __forceinline__ int64_t request_of(const Params &p, int64_t row) {
    int64_t lo = 0, hi = p.num_reqs;  // first b in [0, num_reqs] with cu[b] > row
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(__ldg(p.cu_seqlens_q + mid)) <= row) lo = mid + 1;
        else hi = mid;
    }
    const int64_t b = lo - 1;
    if (b < 0 || b >= p.num_reqs || row >= static_cast<int64_t>(__ldg(p.cu_seqlens_q + b + 1))) return -1;
    return b;
}

__device__ __forceinline__ void row_window(const Params &p, int64_t row, int64_t &n, int64_t &col0) {
    if (p.cu_seqlens_q && request_of(p, row) < 0) {  // no request: an empty row
        n = 0;
        col0 = 0;
        return;
    }
    if (p.seq_lens) {
        const int64_t i = row / p.next_n, t = row % p.next_n;
        const int64_t num = static_cast<int64_t>(__ldg(p.seq_lens + i)) - p.next_n + t + 1;
        n = num <= 0 ? 0 : num / p.compress_ratio;
        if (n > p.width) n = p.width;
        col0 = 0;
    } else {
        const int64_t len = __ldg(p.lengths + row);
        const int64_t rs = p.row_starts ? static_cast<int64_t>(__ldg(p.row_starts + row)) : 0;
        if (rs < 0 || rs > p.width || len <= 0) {
            n = 0;
            col0 = 0;
        } else {
            n = len < p.width - rs ? len : p.width - rs;
            col0 = rs;
        }
    }
}

// Per-row context of the index epilogue: the page-table row and first
// entry (compact page table: the score row and its start; request page
// table: the request, start 0), or the ragged KV offset.
struct RowEpi {
    int64_t pt_row, pt_start;
    int32_t offset;
};

__device__ __forceinline__ RowEpi row_epilogue(const Params &p, int64_t row) {
    RowEpi e{row, 0, 0};
    if (p.idx_offset) e.offset = __ldg(p.idx_offset + row);
    if (p.page_table) {
        if (p.cu_seqlens_q) {
            e.pt_row = request_of(p, row);  // rows no request covers are empty
        } else if (p.pt_row_starts) {
            e.pt_start = __ldg(p.pt_row_starts + row);
        } else if (p.pt_start_is_row_start) {
            e.pt_start = __ldg(p.row_starts + row);
        }
    }
    return e;
}

// The output index of a selected row-local index idx (-1 stays -1): idx
// itself, idx + the ragged offset, or its page-table translation
// page_table[pt_row, pt_start + idx / page_size] * page_size + idx % page_size
// (-1 for a column outside the table; modulo 2^32).
__device__ __forceinline__ int32_t out_index(const Params &p, const RowEpi &e, int32_t idx) {
    if (idx < 0) return -1;
    if (p.idx_offset) return static_cast<int32_t>(static_cast<uint32_t>(idx) + static_cast<uint32_t>(e.offset));
    if (!p.page_table) return idx;
    const int64_t col = e.pt_start + idx / p.page_size;
    if (col < 0 || col >= p.pt_cols) return -1;
    const int64_t page = __ldg(p.page_table + e.pt_row * p.pt_row_stride + col);
    return static_cast<int32_t>(static_cast<uint32_t>(static_cast<uint64_t>(page * p.page_size + idx % p.page_size)));
}

// One output slot j of `row`: the output index, the raw index in out_raw
// (when given), and the value (bit copy, or the dtype's lowest finite value
// for a -1 slot).
template <int DT>
__device__ __forceinline__ void put_mapped(const Params &p, int64_t row, int j, int32_t oi, int32_t idx,
                                           uint32_t raw) {
    using raw_t = typename Elem<DT>::raw_t;
    const int k = p.k;
    p.out_idx[row * k + j] = oi;
    if (p.out_raw) p.out_raw[row * k + j] = idx;
    if (p.out_val)
        static_cast<raw_t *>(p.out_val)[row * k + j] = static_cast<raw_t>(idx >= 0 ? raw : Elem<DT>::kLowest);
}
template <int DT>
__device__ __forceinline__ void put_slot(const Params &p, int64_t row, const RowEpi &e, int j, int32_t idx,
                                         uint32_t raw) {
    put_mapped<DT>(p, row, j, out_index(p, e, idx), idx, raw);
}

template <int DT>
__device__ void emit(const Params &p, int64_t row, const uint2 *sel, int m) {
    const RowEpi ep = row_epilogue(p, row);
    int32_t *orow = p.out_idx + row * p.k;
    if (!p.out_raw && !p.out_val && !p.page_table && !p.idx_offset && m == p.k && (p.k & 3) == 0 &&
        (reinterpret_cast<uintptr_t>(orow) & 15u) == 0u) {
        // four slots per thread and store: 16-byte stores of the column indices
        for (int j = threadIdx.x * 4; j < p.k; j += blockDim.x * 4) {
            const uint4 a = *reinterpret_cast<const uint4 *>(sel + j);
            const uint4 b = *reinterpret_cast<const uint4 *>(sel + j + 2);
            *reinterpret_cast<int4 *>(orow + j) = make_int4(static_cast<int>(a.y), static_cast<int>(a.w),
                                                            static_cast<int>(b.y), static_cast<int>(b.w));
        }
        return;
    }
#pragma unroll 4
    for (int j = threadIdx.x; j < p.k; j += blockDim.x) {
        const bool live = j < m;
        put_slot<DT>(p, row, ep, j, live ? static_cast<int32_t>(sel[j].y) : -1, live ? sel[j].x : 0u);
    }
}

// Order key of a selected (raw, column) pair in the deterministic output:
// (key << 32) | ~column, larger first (value desc, then column asc).
template <int DT>
__device__ __forceinline__ unsigned long long sort_composite(uint2 v) {
    return (static_cast<unsigned long long>(Elem<DT>::key(v.x)) << 32) |
           static_cast<unsigned long long>(0xFFFFFFFFu - v.y);
}

// Deterministic output (value desc, column asc) of the m selected pairs in
// sel, written straight to their output slots.  The keys are counted in
// kBins bins over their own range; a scan from the top gives each bin's
// first slot; the pairs are scattered into their bins' segments (scratch)
// and each pair's slot is its segment's start plus the number of segment
// mates with a larger sort_composite.  Slots m .. k-1 get -1.  `scratch`
// holds kBins counters, then the segments: the composites, the 16-bit
// positions of their pairs in sel and the inverse map (slot -> position),
// or (Compact) the positions alone, the composites being recomputed
// (det_scratch_bytes(sel_cap) bytes in all).  All NT threads call it.
template <int DT, int NT, bool Compact>
__device__ void emit_sorted_impl(const Params &p, int64_t row, const uint2 *sel, int m, uint8_t *scratch,
                                 Ctrl &c, int64_t trace_idx) {
    (void)trace_idx;  // the trace row of this block (GBTOPK_TRACE builds; < 0: none)
    uint32_t *bins = reinterpret_cast<uint32_t *>(scratch);
    unsigned long long *comp = reinterpret_cast<unsigned long long *>(scratch + kBins * 4);
    uint16_t *pos = reinterpret_cast<uint16_t *>(
        scratch + kBins * 4 + (Compact ? 0 : 8 * static_cast<size_t>(p.plan.sel_cap)));
    const int tid = threadIdx.x;
    const RowEpi ep = row_epilogue(p, row);
    if (tid == 0) {
        c.key_min = 0xFFFFFFFFu;
        c.key_max = 0;
    }
    for (int b = tid; b < kBins; b += NT) bins[b] = 0;
    __syncthreads();
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0;
    for (int i = tid; i < m; i += NT) {
        const uint32_t key = Elem<DT>::key(sel[i].x);
        kmin = key < kmin ? key : kmin;
        kmax = key > kmax ? key : kmax;
    }
    block_minmax(kmin, kmax, c);
    if (tid == 0 && trace_idx >= 0) GBTOPK_TRACE_SET(trace_idx, 22, -1);
    if (NT == kFinalThreads && tid == 0) GBTOPK_TRACE_SET(kTraceFinal + blockIdx.x, 3, -1);
    kmin = c.key_min;
    const int bits = 32 - __clz(c.key_max - kmin);
    const int shift = bits > kBinBits ? bits - kBinBits : 0;
    for (int i = tid; i < m; i += NT)
        atomicAdd(&bins[(Elem<DT>::key(sel[i].x) - kmin) >> shift], 1u);
    __syncthreads();
    if (tid == 0 && trace_idx >= 0) GBTOPK_TRACE_SET(trace_idx, 23, -1);
    // bins[b] = pairs in the bins above b
    scan_from_top<NT, kBins>(bins, c, [&](uint32_t b, uint32_t above, uint32_t) { bins[b] = above; });
    if (tid == 0 && trace_idx >= 0) GBTOPK_TRACE_SET(trace_idx, 24, -1);
    if (NT == kFinalThreads && tid == 0) GBTOPK_TRACE_SET(kTraceFinal + blockIdx.x, 4, -1);
    for (int i = tid; i < m; i += NT) {
        const uint2 v = sel[i];
        const uint32_t at = atomicAdd(&bins[(Elem<DT>::key(v.x) - kmin) >> shift], 1u);
        pos[at] = static_cast<uint16_t>(i);
        if constexpr (!Compact) comp[at] = sort_composite<DT>(v);
    }
    __syncthreads();
    if (tid == 0 && trace_idx >= 0) GBTOPK_TRACE_SET(trace_idx, 25, -1);
    if (NT == kFinalThreads && tid == 0) GBTOPK_TRACE_SET(kTraceFinal + blockIdx.x, 5, -1);
    // bins[b] now ends b's segment, which starts where b + 1's ends
    if constexpr (Compact) {
        // rank and write in one pass (no room for an inverse map)
        for (int j = tid; j < m; j += NT) {
            const uint2 v = sel[pos[j]];
            const int32_t oi = out_index(p, ep, static_cast<int32_t>(v.y));  // overlaps the ranking
            const unsigned long long mine = sort_composite<DT>(v);
            const int b = static_cast<int>((static_cast<uint32_t>(mine >> 32) - kmin) >> shift);
            const uint32_t lo = b == kBins - 1 ? 0u : bins[b + 1], hi = bins[b];
            uint32_t before = 0;
            for (uint32_t i = lo; i < hi; ++i) before += sort_composite<DT>(sel[pos[i]]) > mine ? 1u : 0u;
            put_mapped<DT>(p, row, static_cast<int>(lo + before), oi, static_cast<int32_t>(v.y), v.x);
        }
    } else {
        // rank into an inverse map (slot -> position in sel), then write the
        // slots in order: coalesced stores, independent page-table loads
        uint16_t *inv = pos + p.plan.sel_cap;
        for (int j = tid; j < m; j += NT) {
            const unsigned long long mine = comp[j];
            const int b = static_cast<int>((static_cast<uint32_t>(mine >> 32) - kmin) >> shift);
            const uint32_t lo = b == kBins - 1 ? 0u : bins[b + 1], hi = bins[b];
            uint32_t before = 0;
            for (uint32_t i = lo; i < hi; ++i) before += comp[i] > mine ? 1u : 0u;
            inv[lo + before] = pos[j];
        }
        __syncthreads();
        if (tid == 0 && trace_idx >= 0) GBTOPK_TRACE_SET(trace_idx, 26, -1);
        if (NT == kFinalThreads && tid == 0) GBTOPK_TRACE_SET(kTraceFinal + blockIdx.x, 8, -1);
#pragma unroll 4
        for (int j = tid; j < m; j += NT) {
            const uint2 v = sel[inv[j]];
            put_slot<DT>(p, row, ep, j, static_cast<int32_t>(v.y), v.x);
        }
    }
    for (int j = m + tid; j < p.k; j += NT) put_mapped<DT>(p, row, j, -1, -1, 0u);
    __syncthreads();
    if (tid == 0 && trace_idx >= 0) GBTOPK_TRACE_SET(trace_idx, 27, -1);
}

// The sorted output with the segment form the plan's scratch was sized for.
template <int DT, int NT>
__device__ void emit_sorted(const Params &p, int64_t row, const uint2 *sel, int m, uint8_t *scratch, Ctrl &c,
                            int64_t trace_idx = -1) {
    if (p.plan.sel_cap <= kPairSortMax) emit_sorted_impl<DT, NT, false>(p, row, sel, m, scratch, c, trace_idx);
    else emit_sorted_impl<DT, NT, true>(p, row, sel, m, scratch, c, trace_idx);
}

// ---------------------------------------------------------------- bulk staging

// A span of elements staged by one bulk copy: the copy covers the 16-byte
// aligned bytes [a0, a1) around the elements, so element e of the span lands
// at stage[off + e].  The bytes outside the span (at most 15 on each side,
// inside the same allocation) are copied but never used.
struct Span {
    const uint8_t *a0;
    uint32_t bytes;
    int32_t off;
};

template <int DT>
__device__ __forceinline__ Span span_of(const typename Elem<DT>::raw_t *src, int64_t len) {
    constexpr int es = Elem<DT>::kBytes;
    const uintptr_t b = reinterpret_cast<uintptr_t>(src);
    const uintptr_t a0 = b & ~static_cast<uintptr_t>(15);
    const uintptr_t a1 = (b + static_cast<uintptr_t>(len) * es + 15) & ~static_cast<uintptr_t>(15);
    Span sp;
    sp.a0 = reinterpret_cast<const uint8_t *>(a0);
    sp.bytes = static_cast<uint32_t>(a1 - a0);
    sp.off = static_cast<int32_t>((b - a0) / es);
    return sp;
}

// Block-uniform bounded wait on a stage barrier.  On timeout the status
// word is flagged and false is returned (the caller recomputes from global
// memory).
__device__ bool wait_bar(uint8_t *ws, Ctrl &c, unsigned long long *bar, uint32_t parity, uint32_t limit) {
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait(bar, parity, limit);
        c.bcast[7] = ok ? 1u : 0u;
        if (!ok) atomicOr(reinterpret_cast<uint32_t *>(ws), kStatusWaitTimeout);
    }
    __syncthreads();
    const bool ok = c.bcast[7] != 0;
    if (ok) mbar_wait(bar, parity);  // completes at once; acquire for every thread
    return ok;
}

// ---------------------------------------------------------------- element tests

// Element q of a 16-byte vector holding 4 (fp32) or 8 (16-bit) raw values,
// without a dynamically indexed local array.
template <int ES>
__device__ __forceinline__ uint32_t vec_elem(const uint4 &w, int q) {
    if (ES == 4) return q < 2 ? (q == 0 ? w.x : w.y) : (q == 2 ? w.z : w.w);
    const int h = q >> 1;
    const uint32_t word = h < 2 ? (h == 0 ? w.x : w.y) : (h == 2 ? w.z : w.w);
    return (word >> (16 * (q & 1))) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t bin_of(uint32_t key, uint32_t t_lo, int bin_shift) {
    const uint32_t b = (key - t_lo) >> bin_shift;
    return b < static_cast<uint32_t>(kBins - 1) ? b : static_cast<uint32_t>(kBins - 1);
}

// Coarse bin of a candidate key (the top bin takes everything above).
__device__ __forceinline__ uint32_t coarse_bin(uint32_t key, uint32_t t_lo, int coarse_shift) {
    const uint32_t b = (key - t_lo) >> coarse_shift;
    return b < static_cast<uint32_t>(kCoarseBins - 1) ? b : static_cast<uint32_t>(kCoarseBins - 1);
}

__device__ __forceinline__ float float_of_key(uint32_t t) {
    return __uint_as_float((t & 0x80000000u) ? (t & 0x7FFFFFFFu) : ~t);
}

// Threshold test of one raw element: key(raw) >= t_lo.  For fp32 it is one
// float compare against the float whose key is t_lo (signed zeros compare
// equal in IEEE arithmetic, so the two tests agree).
//
// mask(w) tests the 16-byte vector w at once (bit q = element q).  For the
// 16-bit types it compares packed pairs against the raw value whose key is
// t_lo: IEEE order, with signed zeros equal, is the key order.  A compare
// that flushed subnormals to zero could only turn "below" into "equal"
// (flushing is monotone), so it can add candidates but never drop one.
template <int DT>
struct PassTest {
    uint32_t t_lo;
    float tf;
    uint32_t t2;  // 16-bit types: the threshold's raw value in both halves
    __device__ __forceinline__ explicit PassTest(uint32_t t) : t_lo(t), tf(float_of_key(t)) {
        const uint32_t r16 = (t & 0x8000u) ? (t & 0x7FFFu) : (~t & 0xFFFFu);
        t2 = r16 | (r16 << 16);
    }
    __device__ __forceinline__ bool operator()(uint32_t raw) const {
        if (Elem<DT>::kBytes == 4) return __uint_as_float(raw) >= tf;
        return Elem<DT>::key(raw) >= t_lo;
    }
    // 0xFFFF in each half of the packed pair `word` that is >= the threshold
    __device__ __forceinline__ uint32_t pair_ge_mask(uint32_t word) const {
        if constexpr (DT == 1) {
            __nv_bfloat162_raw a, b;
            a.x = static_cast<unsigned short>(word & 0xFFFFu);
            a.y = static_cast<unsigned short>(word >> 16);
            b.x = static_cast<unsigned short>(t2 & 0xFFFFu);
            b.y = static_cast<unsigned short>(t2 >> 16);
            return __hge2_mask(__nv_bfloat162(a), __nv_bfloat162(b));
        } else {
            __half2_raw a, b;
            a.x = static_cast<unsigned short>(word & 0xFFFFu);
            a.y = static_cast<unsigned short>(word >> 16);
            b.x = static_cast<unsigned short>(t2 & 0xFFFFu);
            b.y = static_cast<unsigned short>(t2 >> 16);
            return __hge2_mask(__half2(a), __half2(b));
        }
    }
    __device__ __forceinline__ uint32_t mask(const uint4 &w) const {
        if constexpr (Elem<DT>::kBytes == 4) {
            return static_cast<uint32_t>(__uint_as_float(w.x) >= tf) |
                   (static_cast<uint32_t>(__uint_as_float(w.y) >= tf) << 1) |
                   (static_cast<uint32_t>(__uint_as_float(w.z) >= tf) << 2) |
                   (static_cast<uint32_t>(__uint_as_float(w.w) >= tf) << 3);
        } else {
            // the top byte of each compared half (0xFF or 0) into one byte per
            // element, then the bytes' top bits gathered by one multiply (bits
            // 7, 15, 23, 31 land on 28-31; no two partial products overlap)
            const uint32_t lo = prmt(pair_ge_mask(w.x), pair_ge_mask(w.y), 0x7531u) & 0x80808080u;
            const uint32_t hi = prmt(pair_ge_mask(w.z), pair_ge_mask(w.w), 0x7531u) & 0x80808080u;
            return ((lo * 0x00204081u) >> 28) | (((hi * 0x00204081u) >> 28) << 4);
        }
    }
};

// Lanes of a staged 16-byte vector v that hold elements [0, len) of a span
// whose element 0 sits at element position `off` of the stage.
template <int EPV>
__device__ __forceinline__ uint32_t valid_lanes(int v, int nvec, int off, int len) {
    const int e0 = v * EPV - off;
    const int lo = e0 < 0 ? -e0 : 0;
    const int hi = (len - e0) < EPV ? (len - e0) : EPV;
    return (v < nvec && hi > lo) ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
}

// ---------------------------------------------------------------- threshold guess

// Block-wide suffix search over NB counters: the bin b holding the r-th
// largest item (S(b+1) < r <= S(b), S = count from the top).  Writes b to
// c.bcast[2], the count above it to c.bcast[3] and its own count to
// c.bcast[4].  Requires 1 <= r <= sum of counts.
template <int NT, int NB = kBins>
__device__ void find_bin_from_top(const uint32_t *hist, uint32_t r, Ctrl &c) {
    scan_from_top<NT, NB>(hist, c, [&](uint32_t b, uint32_t above, uint32_t cnt) {
        if (above < r && r <= above + cnt) {
            c.bcast[2] = b;
            c.bcast[3] = above;
            c.bcast[4] = cnt;
        }
    });
}

// Conservative rank-r threshold of m keys in shared memory whose range is
// [kmin, kmax]: a histogram round over NB bins spanning the range (fine
// bins, so the shared-memory increments rarely collide) finds the bin that
// holds the r-th largest key; a second round splits that bin into NB
// sub-bins.  Returns the lower key edge of the sub-bin holding the r-th
// largest key, so at least r keys are >= the result.  Also returns, in
// `upper_e`, the top key of the first-round bin holding the e-th largest
// key (1 <= e <= r): an upper estimate of that key.
// Warp 0: for ranks r0 and r1 (1-based, <= the total count), the bins of
// hist[NB] holding the r0-th and r1-th largest items: c.bcast[2 + 3i] = the
// bin, c.bcast[3 + 3i] = the count above it, c.bcast[4 + 3i] = its count
// (i = 0, 1).  Lane l first sums the run of PER = NB / 32 bins below
// NB - PER l (vector loads) and one warp scan finds the run holding each
// rank; then lane j reads the j-th bin from the top of that run and a
// second warp scan finds the bin (no counter array held per lane).  The
// caller syncs the block after it.
template <int NB>
__device__ __forceinline__ void warp_find_two_bins(const uint32_t *hist, uint32_t r0, uint32_t r1, Ctrl &c) {
    constexpr int PER = NB / 32;
    static_assert(PER % 4 == 0 && PER <= 32, "vector loads, one bin per lane of a run");
    if (threadIdx.x >= 32) return;
    const uint32_t lane = lane_id();
    const uint4 *h4 = reinterpret_cast<const uint4 *>(hist + NB - PER * (static_cast<int>(lane) + 1));
    uint32_t s = 0;
#pragma unroll
    for (int q = 0; q < PER / 4; ++q) {
        const uint4 v = h4[q];
        s += (v.x + v.y) + (v.z + v.w);
    }
    const uint32_t incl = warp_incl_scan(s);
    const uint32_t excl = incl - s;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t r = i == 0 ? r0 : r1;
        const uint32_t bal = __ballot_sync(0xffffffffu, excl < r && r <= incl);
        if (bal == 0u) continue;  // (warp-uniform) r above the total
        const int owner = __ffs(bal) - 1;
        const uint32_t base = __shfl_sync(0xffffffffu, excl, owner);
        const int top = NB - 1 - PER * owner;  // the run's top bin
        const uint32_t cnt = static_cast<int>(lane) < PER ? hist[top - static_cast<int>(lane)] : 0u;
        const uint32_t in2 = base + warp_incl_scan(cnt);
        const uint32_t f = __ffs(__ballot_sync(0xffffffffu, in2 >= r)) - 1;  // a lane < PER
        if (lane == f) {
            c.bcast[2 + 3 * i] = static_cast<uint32_t>(top - static_cast<int>(f));
            c.bcast[3 + 3 * i] = in2 - cnt;
            c.bcast[4 + 3 * i] = cnt;
        }
    }
}

// A sample's keys as one thread holds them: key j is valid for j < count.
struct ThreadKeys {
    static constexpr int kMax = 8;
    uint32_t key[kMax];
    int count;
};

template <int NT, int NB>
__device__ uint32_t adaptive_threshold(const ThreadKeys &tk, uint32_t r, uint32_t e, uint32_t kmin,
                                       uint32_t kmax, uint32_t *hist, Ctrl &c, uint32_t &upper_e) {
    constexpr int NBITS = NB == 512 ? 9 : (NB == 1024 ? 10 : (NB == 2048 ? 11 : 12));
    static_assert((1 << NBITS) == NB, "bin count");
    const int bits = 32 - __clz(kmax - kmin);
    const int shift = bits > NBITS ? bits - NBITS : 0;
#pragma unroll
    for (int j = 0; j < NB / NT; ++j) hist[threadIdx.x + j * NT] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < ThreadKeys::kMax; ++j)
        if (j < tk.count) atomicAdd(&hist[(tk.key[j] - kmin) >> shift], 1u);
    __syncthreads();
    if (threadIdx.x == 0) GBTOPK_TRACE_SET(blockIdx.x, 16, -1);  // (row kernel blocks)
    warp_find_two_bins<NB>(hist, e, r, c);
    __syncthreads();
    if (threadIdx.x == 0) GBTOPK_TRACE_SET(blockIdx.x, 17, -1);
    const uint32_t be = c.bcast[2];
    upper_e = kmin + (be << shift) + ((1u << shift) - 1u);
    if (upper_e < kmin || upper_e > kmax) upper_e = kmax;  // the top bin may reach past kmax
    const uint32_t b = c.bcast[5];
    const uint32_t rem = r - c.bcast[6];
    const uint32_t edge = kmin + (b << shift);
    if (shift == 0 || c.bcast[7] == rem) return edge;  // exact key, or the whole bin is needed
    const int shift2 = shift > NBITS ? shift - NBITS : 0;
#pragma unroll
    for (int j = 0; j < NB / NT; ++j) hist[threadIdx.x + j * NT] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < ThreadKeys::kMax; ++j) {
        const uint32_t d = tk.key[j] - kmin;
        if (j < tk.count && (d >> shift) == b) atomicAdd(&hist[(d - (b << shift)) >> shift2], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) GBTOPK_TRACE_SET(blockIdx.x, 18, -1);
    warp_find_two_bins<NB>(hist, rem, rem, c);
    __syncthreads();
    return edge + (c.bcast[2] << shift2);
}

// The value whose key (Elem<DT>::key) is `key`, widened to float (exact for
// every value of the three types; both zeros give +0).
template <int DT>
__device__ __forceinline__ float key_value(uint32_t key) {
    if constexpr (DT == 0) {
        return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
    } else {
        const uint32_t raw = (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
        if constexpr (DT == 1) {
            return __uint_as_float(raw << 16);
        } else {
            return __half2float(__ushort_as_half(static_cast<unsigned short>(raw)));
        }
    }
}

// The key of value v rounded down (up) to the element type: every element
// whose value is >= v (<= v) has a key >= (<=) the result.
template <int DT>
__device__ __forceinline__ uint32_t key_of_value(float v, bool up) {
    if constexpr (DT == 0) {
        return Elem<DT>::key(__float_as_uint(v));
    } else if constexpr (DT == 1) {
        const __nv_bfloat16 h = up ? __float2bfloat16_ru(v) : __float2bfloat16_rd(v);
        return Elem<DT>::key(__bfloat16_as_ushort(h));
    } else {
        const __half h = up ? __float2half_ru(v) : __float2half_rd(v);
        return Elem<DT>::key(__half_as_ushort(h));
    }
}

// Conservative rank-r threshold of the sample over bins of equal VALUE
// width: NB bins spanning the sample's value range [value(kmin),
// value(kmax)].  The bin of a key is a nondecreasing function of its value
// (rounded subtract, multiply and truncation are all monotone), and key
// order is value order.  Warp 0 finds the bins holding the e-th and r-th
// largest keys; the threshold is the key of the r-th's bin's lower value
// edge less half a bin (the margin covers the rounding of the bin map, so
// at least r keys are >= it), the upper estimate of the e-th key that of
// its bin's upper edge.  Where the sample is dense, value bins hold a few
// keys each, while bins of equal key width follow the binades and crowd
// the sample into a few dozen bins, so one round here does the work of
// adaptive_threshold's two.  That function is still taken when the value
// range is not a finite positive span at least 1/256 of the largest
// magnitude (where the half-bin margin would not cover the rounding), or
// when the r-th's bin holds more than max(16, r / 8) keys (a wide range
// around a dense cluster), which would leave the threshold too far below
// the r-th key.
template <int DT, int NT, int NB>
__device__ uint32_t value_threshold(const ThreadKeys &tk, uint32_t r, uint32_t e, uint32_t kmin, uint32_t kmax,
                                    uint32_t *hist, Ctrl &c, uint32_t &upper_e) {
    constexpr float kFltMax = 3.402823466e38f;
    const float vmin = key_value<DT>(kmin);
    const float vmax = key_value<DT>(kmax);
    const float span = __fsub_rn(vmax, vmin);
    const float scale = span > 0.0f ? __fdiv_rn(static_cast<float>(NB), span) : 0.0f;
    const float amax = fmaxf(fabsf(vmin), fabsf(vmax));
    // block-uniform from here on
    bool by_keys = !(span > 0.0f && span <= kFltMax && scale > 0.0f && scale <= kFltMax &&
                     span >= amax * (1.0f / 256.0f));
    uint32_t t = 0;
    if (!by_keys) {
#pragma unroll
        for (int j = 0; j < NB / NT; ++j) hist[threadIdx.x + j * NT] = 0;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < ThreadKeys::kMax; ++j) {
            if (j < tk.count) {
                const int q = __float2int_rz(__fmul_rn(__fsub_rn(key_value<DT>(tk.key[j]), vmin), scale));
                atomicAdd(&hist[q < 0 ? 0 : (q > NB - 1 ? NB - 1 : q)], 1u);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) GBTOPK_TRACE_SET(blockIdx.x, 16, -1);  // (row kernel blocks)
        warp_find_two_bins<NB>(hist, e, r, c);
        __syncthreads();
        if (threadIdx.x == 0) GBTOPK_TRACE_SET(blockIdx.x, 17, -1);
        const uint32_t be = c.bcast[2];
        const uint32_t b = c.bcast[5];
        const uint32_t lim = r / 8u > 16u ? r / 8u : 16u;
        by_keys = c.bcast[7] > lim;
        if (!by_keys) {
            const float bw = span * (1.0f / static_cast<float>(NB));  // bin width
            t = key_of_value<DT>(vmin + (static_cast<float>(b) - 0.5f) * bw, false);
            if (t < kmin) t = kmin;
            uint32_t u = key_of_value<DT>(vmin + (static_cast<float>(be) + 1.0f) * bw, true);
            if (u > kmax) u = kmax;
            upper_e = u > t ? u : t;
        }
    }
    if (by_keys) t = adaptive_threshold<NT, NB>(tk, r, e, kmin, kmax, hist, c, upper_e);
    return t;
}

// The guess from a sample of m keys (with their min and max) of a row of n
// columns: t_lo such that, with high probability, at least k row elements
// are >= t_lo (the sample rank r = e + 6 sqrt(e) + 2, e = m k / n); and the
// histogram scale of the candidates: keys t_lo .. t_est map onto the lower
// half of kBins, t_est being an upper estimate of the sample's e-th key
// (where the k-th key of the row is expected), so the k-th key lands in
// fine bins even when the keys above it span many binades or both signs;
// keys far above it pile into the top bins, which are taken whole.
template <int DT, int NT>
__device__ void guess_from_sample(const ThreadKeys &sample, int m, int64_t n, int k, uint32_t kmin,
                                  uint32_t kmax, uint32_t *hist, Ctrl &c, uint32_t &t_lo,
                                  int &bin_shift, int &coarse_shift) {
    uint32_t r = guess_rank(n, k);
    if (r > static_cast<uint32_t>(m)) r = static_cast<uint32_t>(m);
    uint32_t e = static_cast<uint32_t>((static_cast<int64_t>(m) * k + n - 1) / n);
    e = e < 1u ? 1u : (e > r ? r : e);
    uint32_t t_est;
    t_lo = value_threshold<DT, NT, kGuessBins>(sample, r, e, kmin, kmax, hist, c, t_est);
    const int bits = 32 - __clz(t_est - t_lo);
    bin_shift = bits > kBinBits - 1 ? bits - (kBinBits - 1) : 0;
    constexpr int kCoarseBits = 8;  // log2(kCoarseBins)
    static_assert((1 << kCoarseBits) == kCoarseBins, "coarse bins");
    coarse_shift = bits > kCoarseBits - 1 ? bits - (kCoarseBits - 1) : 0;
}


// ---------------------------------------------------------------- block filter

// Keeps the staged elements [off, off + len) of `stage` whose key is >= t_lo.
// Each thread loads its vectors (strided by the block size) into registers
// and marks passing elements in bit masks; one block scan then gives each
// thread its output slot, so candidates are written without per-element
// atomics.  put(slot, raw, col) stores one candidate (col = col_base + e).
// Returns the candidate count (block-uniform).  The staged bytes may be
// overwritten by put() (every thread holds its vectors by then).
template <int DT, int VPT, class Put>
__device__ uint32_t filter_staged(const void *stage, int off, int len, int col_base, uint32_t t_lo,
                                  Ctrl &c, Put &&put) {
    constexpr int es = Elem<DT>::kBytes;
    constexpr int EPV = 16 / es;
    const int nvec = ((off + len) * es + 15) >> 4;
    const uint4 *svec = static_cast<const uint4 *>(stage);
    uint4 w[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = threadIdx.x + j * static_cast<int>(blockDim.x);
        w[j] = v < nvec ? svec[v] : make_uint4(0, 0, 0, 0);
    }
    const PassTest<DT> pass(t_lo);
    uint32_t msk[VPT];
    uint32_t cnt = 0;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = threadIdx.x + j * static_cast<int>(blockDim.x);
        msk[j] = pass.mask(w[j]) & valid_lanes<EPV>(v, nvec, off, len);
        cnt += __popc(msk[j]);
    }
    uint32_t total;
    uint32_t slot = block_excl_scan(cnt, c, total);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        uint32_t m = msk[j];
        const int v = threadIdx.x + j * static_cast<int>(blockDim.x);
        while (m) {
            const int q = __ffs(m) - 1;
            m &= m - 1;
            put(slot++, vec_elem<es>(w[j], q), static_cast<uint32_t>(col_base + v * EPV + q - off));
        }
    }
    return total;
}

// Places the best `need` of the bsize members of blist (shared memory) at
// sel[above + rank], rank being the member's position in the total order
// (key desc, then the tie mode's column order; smaller columns first for
// tie mode 0), which no two members share.  Each member's order is packed
// into one 64-bit composite (key above, complemented tie column below),
// blist is overwritten with the composites, and each member is ranked by
// counting the composites above its own.  All threads; ends with a barrier.
template <int DT>
__device__ void rank_all(uint2 *blist, uint32_t bsize, uint32_t need, uint32_t above, int tie, uint2 *sel) {
    unsigned long long *comp = reinterpret_cast<unsigned long long *>(blist);
    constexpr int kMaxPer = 4;  // members per thread (bsize <= 4 * blockDim.x)
    uint2 me[kMaxPer];
    unsigned long long mine[kMaxPer];
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q) {
        const uint32_t i = threadIdx.x + q * blockDim.x;
        me[q] = i < bsize ? blist[i] : make_uint2(0u, 0u);
        mine[q] = (static_cast<unsigned long long>(Elem<DT>::key(me[q].x)) << 32) | ~tie_key(me[q].y, tie);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q) {
        const uint32_t i = threadIdx.x + q * blockDim.x;
        if (i < bsize) comp[i] = mine[q];
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q) {
        const uint32_t i = threadIdx.x + q * blockDim.x;
        if (i < bsize) {
            uint32_t rank = 0;
#pragma unroll 4
            for (uint32_t j = 0; j < bsize; ++j) rank += comp[j] > mine[q] ? 1u : 0u;
            if (rank < need) sel[above + rank] = me[q];
        }
    }
    __syncthreads();
}

// Finds the exact top-k among `total` (>= k) candidates whose keys are
// counted in hist[kBins] (shared memory): the bin b* holding the k-th key
// from the top, every candidate of a higher bin, and the best `need` of bin
// b* (ranked by key, then by smaller column).  Writes sel[0..k).  Returns
// false when bin b* holds more candidates than `bcap` (caller falls back).
// `sel` may alias `hist` (the histogram is consumed first).
template <int DT, int NT, class CandSrc>
__device__ bool select_from_candidates(const CandSrc &cands, uint32_t total, const uint32_t *hist,
                                       uint32_t t_lo, int bin_shift, int k, int tie, uint2 *sel,
                                       uint2 *blist, uint32_t bcap, Ctrl &c) {
    constexpr int KB = Elem<DT>::kKeyBits;
    find_bin_from_top<NT>(hist, static_cast<uint32_t>(k), c);
    if (threadIdx.x == 0) {
        c.sel_count = 0;
        c.b_count = 0;
    }
    __syncthreads();
    const uint32_t bstar = c.bcast[2], above = c.bcast[3], bsize = c.bcast[4];
    if (bsize > bcap) return false;
    for_each_item(cands, total, [&](bool valid, uint32_t key, uint32_t idx, uint32_t raw) {
        const uint32_t b = bin_of(key, t_lo, bin_shift);
        const bool hi = valid && b > bstar;
        const bool eq = valid && b == bstar;
        const uint32_t slot = warp_claim(&c.sel_count, hi);
        if (hi) sel[slot] = make_uint2(raw, idx);
        const uint32_t bslot = warp_claim(&c.b_count, eq);
        if (eq) blist[bslot] = make_uint2(raw, idx);
    });
    __syncthreads();
    const uint32_t need = static_cast<uint32_t>(k) - above;
    if (bsize <= kRankMax) {
        rank_all<DT>(blist, bsize, need, above, tie, sel);
    } else {
        const PairSrc<DT> bs{blist};
        uint32_t t, gt;
        block_select<KB, KB / 8>(bs, RankByKey{}, bsize, need, c.rhist, c, t, gt);
        const uint32_t need_ties = need - gt;
        uint32_t col_max = 0xFFFFFFFFu;
        if (tie) {
            uint32_t kk, g2;
            block_select<32, 4>(bs, RankTieColumn{t, tie}, bsize, need_ties, c.rhist, c, kk, g2);
            col_max = ~kk;
        }
        collect<DT>(bs, bsize, t, gt, need_ties, tie, col_max, sel, above, c);
    }
    return true;
}

// ---------------------------------------------------------------- workspace layout

__device__ __forceinline__ uint8_t *row_ws(const Params &p, int64_t row) {
    return p.ws + kWsHeaderBytes + static_cast<size_t>(row) * p.plan.ws_row_bytes;
}
__device__ __forceinline__ uint32_t *row_info(const Params &p, int64_t row) {
    return reinterpret_cast<uint32_t *>(row_ws(p, row));
}
__device__ __forceinline__ uint32_t *row_counts(const Params &p, int64_t row) {
    return reinterpret_cast<uint32_t *>(row_ws(p, row) + kRowInfoBytes);
}
__device__ __forceinline__ uint32_t *row_hist(const Params &p, int64_t row) {
    return reinterpret_cast<uint32_t *>(row_ws(p, row) + ws_hist_offset(p.plan.chunks_per_row));
}
__device__ __forceinline__ uint2 *row_segs(const Params &p, int64_t row) {
    return reinterpret_cast<uint2 *>(row_ws(p, row) + ws_seg_offset(p.plan.chunks_per_row));
}

__device__ __forceinline__ int64_t split_chunks(const Params &p, int64_t n) {
    return n > p.plan.direct_max ? (n + p.plan.chunk - 1) / p.plan.chunk : 0;
}

// ---------------------------------------------------------------- kernels

// Row kernel: one block per row.  Empty and short rows (n <= k) and rows up
// to direct_max columns are finished here (the row is staged in shared
// memory by one bulk copy).  For longer rows it computes the threshold guess
// from a strided sample (256 groups of 8 consecutive columns) and stores it
// in the row's workspace for the stream and finalize kernels.  It releases
// the dependent stream kernel (programmatic dependent launch) once its own
// global loads are in, so the stream's bulk copies do not queue ahead of them.
// Narrow variants (VPT <= 3) keep to 64 registers so four blocks share an SM.
template <int DT, int VPT>
__global__ void __launch_bounds__(kThreads, VPT <= 3 ? 4 : 1) row_kernel(const __grid_constant__ Params p) {
    using raw_t = typename Elem<DT>::raw_t;
    extern __shared__ __align__(128) uint8_t smem[];
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + p.plan.off_hist);
    uint2 *sel = reinterpret_cast<uint2 *>(smem + p.plan.off_hist);  // aliases hist
    // after the guess's counters; dead once the guess is made (direct rows
    // then zero the whole histogram over it)
    uint32_t *sample = reinterpret_cast<uint32_t *>(smem + p.plan.off_hist + kGuessBins * 4);
    uint8_t *stage = smem + p.plan.off_stage;  // direct rows; the sorted output's scratch
    const int64_t row = p.row0 + blockIdx.x;
    const int k = p.k;
    const bool sorted = sorted_output(p.deterministic);
    const int tie = tie_mode(p.deterministic);
    constexpr int kTraceBase = 0;
    (void)kTraceBase;

    GBTOPK_TRACE_POINT(0, 0);
    // launched as a programmatic dependent of whatever ran before on the
    // stream: no input is read before that kernel has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int64_t n, col0;
    row_window(p, row, n, col0);
    const raw_t *xrow = static_cast<const raw_t *>(p.x) + row * p.row_stride + col0;
    if (threadIdx.x == 0) {
        c.key_min = 0xFFFFFFFFu;
        c.key_max = 0;
        // this call's stream abort word, read by the finalize kernel once
        // the stream kernel has completed
        if (p.plan.split && blockIdx.x == 0) reinterpret_cast<uint32_t *>(p.ws)[1] = 0;
    }

    if (n > p.plan.direct_max) {
        // the chunk / stream kernel may launch at once: its bulk copies of the
        // row then overlap this guess (it reads the guess only once this grid
        // has completed)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // ---- split row: threshold guess from a strided sample (the whole
        // row when it has at most kSampleSize columns).  First clear the
        // row's coarse candidate histogram, which the chunk kernel counts
        // into once this grid has completed.
        if (threadIdx.x < kCoarseBins / 4)
            reinterpret_cast<uint4 *>(row_hist(p, row))[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
        int m;
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0;
        ThreadKeys tk;  // this thread's sample keys (registers)
        // hint anchor (the previous argmax column): thread 32 issues its two
        // dependent loads alongside the sample's, and folds the value in
        // after the barrier
        constexpr int kHintThread = 32;
        int32_t a = -1;
        if (threadIdx.x == kHintThread && p.pre_idx) a = __ldg(p.pre_idx + (row / p.next_n) * k);
        if (n > kSampleSize) {
            m = kSampleSize;
            // group of 8 consecutive columns, moved down to a 16-byte
            // boundary (one or two vector loads) unless that would leave the row
            int64_t pos = static_cast<int64_t>(threadIdx.x) * (n - 8) / (kSampleGroups - 1);
            const uintptr_t addr = reinterpret_cast<uintptr_t>(xrow + pos);
            const int64_t back = static_cast<int64_t>((addr & 15u) / Elem<DT>::kBytes);
            uint32_t raw[8];
            if (back <= pos) {
                pos -= back;
                const uint4 *v = reinterpret_cast<const uint4 *>(xrow + pos);
                if constexpr (Elem<DT>::kBytes == 4) {
                    const uint4 a = __ldg(v), b = __ldg(v + 1);
                    raw[0] = a.x; raw[1] = a.y; raw[2] = a.z; raw[3] = a.w;
                    raw[4] = b.x; raw[5] = b.y; raw[6] = b.z; raw[7] = b.w;
                } else {
                    const uint4 a = __ldg(v);
                    const uint32_t wd[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) raw[j] = (wd[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) raw[j] = ldg_raw(xrow + pos + j);
            }
            static_assert(ThreadKeys::kMax == 8 && kSampleGroups == kThreads, "one group of 8 per thread");
            tk.count = 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t key = Elem<DT>::key(raw[j]);
                tk.key[j] = key;
                kmin = key < kmin ? key : kmin;
                kmax = key > kmax ? key : kmax;
            }
        } else {
            m = static_cast<int>(n);  // the whole row: column threadIdx.x + j kThreads
            static_assert(ThreadKeys::kMax * kThreads >= kSampleSize, "the sample fits the threads' keys");
            tk.count = 0;
#pragma unroll
            for (int j = 0; j < ThreadKeys::kMax; ++j) {
                const int i = static_cast<int>(threadIdx.x) + j * kThreads;
                tk.key[j] = 0u;
                if (i < m) {
                    const uint32_t key = Elem<DT>::key(ldg_raw(xrow + i));
                    tk.key[j] = key;
                    tk.count = j + 1;
                    kmin = key < kmin ? key : kmin;
                    kmax = key > kmax ? key : kmax;
                }
            }
        }
        const bool hint_ok = threadIdx.x == kHintThread &&
                             static_cast<uint64_t>(static_cast<uint32_t>(a)) < static_cast<uint64_t>(n);
        uint32_t hraw = 0;
        if (hint_ok) hraw = ldg_raw(xrow + a);
        __syncthreads();
        GBTOPK_TRACE_POINT(1, 0);
        if (hint_ok) {
            const uint32_t key = Elem<DT>::key(hraw);
            kmax = key > kmax ? key : kmax;
        }
        block_minmax(kmin, kmax, c);
        GBTOPK_TRACE_POINT(2, 0);
        uint32_t t_lo;
        int bin_shift;
        int coarse_shift;
        guess_from_sample<DT, kThreads>(tk, m, n, k, c.key_min, c.key_max, hist, c, t_lo, bin_shift, coarse_shift);
        (void)bin_shift;
        if (threadIdx.x == 0) {
            uint32_t *info = row_info(p, row);
            info[0] = t_lo;
            info[1] = static_cast<uint32_t>(coarse_shift);
            info[2] = 0;  // the row's chunk ticket (fused plans)
        }
        GBTOPK_TRACE_POINT(6, 0);
        GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | 3u);
        GBTOPK_TRACE_ANCHOR();
        return;
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- short and empty rows: every valid column, then -1
    if (n <= k) {
        if (sorted) {
            for (int j = threadIdx.x; j < n; j += blockDim.x)
                sel[j] = make_uint2(ldg_raw(xrow + j), static_cast<uint32_t>(j));
            __syncthreads();
            emit_sorted<DT, kThreads>(p, row, sel, static_cast<int>(n), stage, c);
        } else {
            const RowEpi ep = row_epilogue(p, row);
            for (int j = threadIdx.x; j < k; j += blockDim.x) {
                const bool live = j < n;
                put_slot<DT>(p, row, ep, j, live ? j : -1, live && p.out_val ? ldg_raw(xrow + j) : 0u);
            }
        }
        GBTOPK_TRACE_POINT(6, 0);
        GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | 1u);
        GBTOPK_TRACE_ANCHOR();
        return;
    }

    // ---- direct rows: stage the row, then guess, filter and select in shared memory
    if constexpr (VPT == 0) {
        return;  // split plans: every row longer than top_k went to the guess above
    } else {
    const uint32_t stage_pairs = static_cast<uint32_t>((p.plan.row_smem - p.plan.off_stage) / sizeof(uint2));
    if (threadIdx.x == 0) mbar_init(&c.bar);
    __syncthreads();
    const Span sp = span_of<DT>(xrow, n);
    if (threadIdx.x == 0) bulk_load(stage, sp.a0, sp.bytes, &c.bar);
    const bool ok = wait_bar(p.ws, c, &c.bar, 0, p.wait_polls);
    __syncthreads();
    GBTOPK_TRACE_POINT(3, 0);
    const raw_t *srow = reinterpret_cast<const raw_t *>(stage) + sp.off;
    bool done = false;
    if (ok) {
        const int m = n < kSampleSize ? static_cast<int>(n) : kSampleSize;
        // n <= two chunks (< 2^16 columns): 16.16 fixed point positions are exact enough
        const uint32_t stride = static_cast<uint32_t>((static_cast<uint64_t>(n) << 16) / m);
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0;
        for (int i = threadIdx.x; i < m; i += blockDim.x) {
            const uint32_t key = Elem<DT>::key(srow[(static_cast<uint64_t>(i) * stride) >> 16]);
            sample[i] = key;
            kmin = key < kmin ? key : kmin;
            kmax = key > kmax ? key : kmax;
        }
        block_minmax(kmin, kmax, c);  // (its barrier publishes the sample)
        ThreadKeys tk;
        tk.count = 0;
#pragma unroll
        for (int j = 0; j < ThreadKeys::kMax; ++j) {
            const int i = static_cast<int>(threadIdx.x) + j * kThreads;
            tk.key[j] = i < m ? sample[i] : 0u;
            if (i < m) tk.count = j + 1;
        }
        uint32_t t_lo;
        int bin_shift;
        int coarse_shift;
        guess_from_sample<DT, kThreads>(tk, m, n, k, c.key_min, c.key_max, hist, c, t_lo, bin_shift, coarse_shift);
        (void)coarse_shift;
#pragma unroll
        for (int j = 0; j < kBins / kThreads; ++j) hist[threadIdx.x + j * kThreads] = 0;
        __syncthreads();
        uint2 *lcand = reinterpret_cast<uint2 *>(stage);  // the row is in registers by then
        const uint32_t total = filter_staged<DT, VPT>(
            stage, sp.off, static_cast<int>(n), 0, t_lo, c, [&](uint32_t slot, uint32_t raw, uint32_t col) {
                if (slot < stage_pairs) lcand[slot] = make_uint2(raw, col);
                atomicAdd(&hist[bin_of(Elem<DT>::key(raw), t_lo, bin_shift)], 1u);
            });
        __syncthreads();
        if (total >= static_cast<uint32_t>(k) && total <= stage_pairs)
            done = select_from_candidates<DT, kThreads>(PairSrc<DT>{lcand}, total, hist, t_lo, bin_shift,
                                                        k, tie, sel, lcand + total, stage_pairs - total, c);
    }
    if (!done) exact_select<DT>(GlobalSrc<DT>{xrow}, n, k, tie, sel, c.rhist, c);
    bool stage_ok = ok;
    if (!ok) {  // let the copy land before the stage is reused (bounded)
        if (threadIdx.x == 0) {
            const bool landed = mbar_wait(&c.bar, 0);
            c.bcast[7] = landed ? 1u : 0u;
            if (!landed) atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusCopyLost);
        }
        __syncthreads();
        stage_ok = c.bcast[7] != 0;
    }
    if (sorted && stage_ok) {
        __syncthreads();
        emit_sorted<DT, kThreads>(p, row, sel, k, stage, c);  // the stage is free once the row is selected
    } else {
        emit<DT>(p, row, sel, k);  // the selected set, unordered if the stage was unusable
    }
    GBTOPK_TRACE_POINT(6, 0);
    GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | 2u);
    GBTOPK_TRACE_ANCHOR();
    }
}

// Stream kernel: persistent blocks (one per SM) walk the chunks of the split
// rows, block b taking chunks b, b + G, b + 2G, ... of the dense row-major
// chunk list.  Warp 0 is the producer: it maps chunks to rows and issues
// their bulk copies into a ring of kStages shared-memory stages ("full"
// barriers carry the byte counts).  The other warps are consumers, one group
// per chunk: each loads its slice of the stage into registers, keeps the
// elements at or above the row's guess and appends them to that chunk's
// fixed segment in the workspace (one shared atomic per warp reserves the
// slots; the values are read back from the stage), then releases the stage
// ("empty" barrier); the last warp to finish a chunk stores its count.
// Three 64 KB stages per SM measured faster than six of 32 KB or four of
// 48 KB (fewer, larger copies).  There is no block-wide barrier in the
// steady state.
struct StageMeta {
    int64_t c0;       // first column of the chunk
    int32_t row;      // row index within this launch
    int32_t len;
    int32_t off;
    int32_t seg_cap;
    int32_t chunk;
    int32_t pad;
};

struct RowFacts {
    uint32_t prefix;   // dense number of the row's first chunk
    int32_t n;         // valid columns
    int32_t col0;      // column of local index 0
    uint32_t t_lo;     // threshold guess (after the row kernel)
};
static_assert(sizeof(RowFacts) == 16, "row facts");
static_assert(sizeof(Ctrl) + kStages * sizeof(StageMeta) <= kCtrlBytes, "stage metadata after the control block");

__device__ __forceinline__ void mbar_init_count(unsigned long long *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(kStreamThreads) stream_kernel(const __grid_constant__ Params p) {
    using raw_t = typename Elem<DT>::raw_t;
    constexpr int es = Elem<DT>::kBytes;
    constexpr int EPV = 16 / es;
    constexpr int NCW = kStreamThreads / 32 - 1;  // consumer warps
    constexpr int kGroups = NCW / kGroupWarps;      // consumer groups take chunks in turn
    constexpr int VPL = (kChunkBytes + 16) / 16 / (kGroupWarps * 32) + 1;
    static_assert(kStages % kGroups == 0, "each group cycles its own stages");
    extern __shared__ __align__(128) uint8_t smem[];
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem);
    const int rows = static_cast<int>(p.rows);
    RowFacts *rf = reinterpret_cast<RowFacts *>(smem + kCtrlBytes);  // rows + 1 entries
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + kCtrlBytes - kStages * sizeof(StageMeta));
    uint8_t *stages = smem + p.plan.stream_smem - static_cast<size_t>(kStages) * kStageBytes;
    const int64_t CH = p.plan.chunk;
    constexpr int kTraceBase = kTraceStream;
    (void)kTraceBase;
    GBTOPK_TRACE_POINT(0, 0);

    // dense numbering of the chunks of the split rows of this launch
    constexpr int RPT = (kMaxBlockRows + kStreamThreads - 1) / kStreamThreads;
    uint32_t nch_local[RPT], sum = 0;
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int r = threadIdx.x * RPT + j;
        uint32_t nc = 0;
        if (r < rows) {
            int64_t n, col0;
            row_window(p, p.row0 + r, n, col0);
            nc = static_cast<uint32_t>(split_chunks(p, n));
            rf[r].n = static_cast<int32_t>(n);
            rf[r].col0 = static_cast<int32_t>(col0);
        }
        nch_local[j] = nc;
        sum += nc;
    }
    uint32_t total_items;
    uint32_t acc = block_excl_scan(sum, c, total_items);
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int r = threadIdx.x * RPT + j;
        if (r <= rows) rf[r].prefix = acc;
        acc += nch_local[j];
    }
    if (threadIdx.x == 0) {
        rf[rows].prefix = total_items;
        c.abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init_count(&c.full[s], 1);
            mbar_init_count(&c.empty[s], kGroupWarps);
            c.scombo[0][s] = c.scombo[1][s] = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int64_t G = gridDim.x;
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
#ifdef GBTOPK_TRACE
            unsigned long long p_wait = 0;
#endif
            int64_t issued = 0;
            bool aborted = false;
            for (int64_t i = 0;; ++i) {
                const int64_t item = blockIdx.x + i * G;
                if (item >= total_items) break;
                const int s = static_cast<int>(i % kStages);
                if (i >= kStages) {
                    const uint32_t par = static_cast<uint32_t>(((i / kStages) - 1) & 1);
#ifdef GBTOPK_TRACE
                    const unsigned long long pa = clock64();
#endif
                    const int got = mbar_wait_or_abort(&c.empty[s], par, p.wait_polls, &c.abort_flag);
#ifdef GBTOPK_TRACE
                    p_wait += clock64() - pa;
#endif
                    if (got != 1) {  // stop streaming: the consumers stop too
                        atomicExch(&c.abort_flag, 1u);
                        atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusWaitTimeout);
                        aborted = true;
                        break;
                    }
                }
                int lo = 0, hi = rows - 1;  // last row with prefix <= item
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (rf[mid].prefix <= item) lo = mid;
                    else hi = mid - 1;
                }
                const RowFacts f = rf[lo];
                const int64_t chunk = item - f.prefix;
                const int64_t c0 = chunk * CH;
                const int64_t len = (f.n - c0) < CH ? (f.n - c0) : CH;
                const raw_t *src =
                    static_cast<const raw_t *>(p.x) + (p.row0 + lo) * p.row_stride + f.col0 + c0;
                const Span sp = span_of<DT>(src, len);
                StageMeta &m = meta[s];
                m.c0 = c0;
                m.row = lo;
                m.len = static_cast<int32_t>(len);
                m.off = sp.off;
                m.chunk = static_cast<int32_t>(chunk);
                m.seg_cap = chunk_seg_cap(f.n, p.k, p.plan.chunk);
                bulk_load(stages + static_cast<size_t>(s) * kStageBytes, sp.a0, sp.bytes, &c.full[s]);
                issued = i + 1;
            }
#ifdef GBTOPK_TRACE
            if (kTraceBase + blockIdx.x < kTraceBlocks) g_trace[kTraceBase + blockIdx.x][12] = p_wait;
#endif
            c.bcast[0] = static_cast<uint32_t>(issued);  // for the drain below
            (void)aborted;
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
    } else {
        // ---- consumers: the row kernel's guesses (programmatic dependent launch)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int r = threadIdx.x - 32; r < rows; r += NCW * 32)
            if (rf[r].n > p.plan.direct_max) rf[r].t_lo = __ldcg(row_info(p, p.row0 + r));
        asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");

        const int cw = warp - 1;
        const int grp = cw / kGroupWarps, gw = cw % kGroupWarps;
        const int my_items = blockIdx.x < total_items
                                 ? static_cast<int>((total_items - blockIdx.x + G - 1) / G) : 0;
    #ifdef GBTOPK_TRACE
        unsigned long long t_wait = 0, t_busy = 0, t_mark = clock64(), n_items = 0;
    #endif
        for (int i = grp; i < my_items; i += kGroups) {
            const int s = i % kStages;
            const uint32_t par = static_cast<uint32_t>((i / kStages) & 1);
    #ifdef GBTOPK_TRACE
            unsigned long long t_a = clock64();
            t_busy += t_a - t_mark;
    #endif
            // a stage the producer never filled must not be read, nor its
            // metadata: on a timeout or an abort the warp stops, and the
            // finalize kernel recomputes every row of the call from global memory
            int got = 0;
            if (lane == 0) got = mbar_wait_or_abort(&c.full[s], par, p.wait_polls, &c.abort_flag);
            got = __shfl_sync(0xffffffffu, got, 0);
    #ifdef GBTOPK_TRACE
            t_mark = clock64();
            t_wait += t_mark - t_a;
            ++n_items;
    #endif
            if (got != 1) {
                if (got == 0 && lane == 0) {
                    atomicExch(&c.abort_flag, 1u);
                    atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusWaitTimeout);
                    reinterpret_cast<volatile uint32_t *>(p.ws)[1] = 1u;
                }
                break;
            }
            mbar_wait(&c.full[s], par);  // completes at once: acquire for every lane
            const StageMeta m = meta[s];
            const int64_t grow = p.row0 + m.row;
            const int nvec = ((m.off + m.len) * es + 15) >> 4;
            const uint4 *svec = reinterpret_cast<const uint4 *>(stages + static_cast<size_t>(s) * kStageBytes);
            const int vbase = gw * 32 + static_cast<int>(lane);
            uint4 w[VPL];
    #pragma unroll
            for (int j = 0; j < VPL; ++j) {
                const int v = vbase + j * kGroupWarps * 32;
                w[j] = v < nvec ? svec[v] : make_uint4(0, 0, 0, 0);
            }
            const PassTest<DT> pass(rf[m.row].t_lo);
            uint32_t msk[VPL];
            uint32_t cnt = 0;
    #pragma unroll
            for (int j = 0; j < VPL; ++j) {
                const int v = vbase + j * kGroupWarps * 32;
                uint32_t bits = pass.mask(w[j]);
                if (v == 0 || v >= nvec - 1) bits &= valid_lanes<EPV>(v, nvec, m.off, m.len);
                msk[j] = bits;
                cnt += __popc(bits);
            }
            // warp-level slot reservation; the same atomic counts the warps done
            uint32_t incl = cnt;
    #pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= static_cast<uint32_t>(o)) incl += y;
            }
            const uint32_t wtotal = __shfl_sync(0xffffffffu, incl, 31);
            unsigned long long old = 0;
            if (lane == 0) old = atomicAdd(&c.scombo[par][s], (1ull << 32) | wtotal);
            const uint32_t base = __shfl_sync(0xffffffffu, static_cast<uint32_t>(old), 0);
            if (lane == 0 && static_cast<uint32_t>(old >> 32) == kGroupWarps - 1) {  // last warp on the chunk
                row_counts(p, grow)[m.chunk] = base + wtotal;
                c.scombo[par][s] = 0;
            }
            uint32_t slot = base + incl - cnt;
            const uint32_t cap = static_cast<uint32_t>(m.seg_cap);
            uint2 *seg = row_segs(p, grow) + static_cast<int64_t>(m.chunk) * m.seg_cap;
            const int colbase = static_cast<int>(m.c0) - m.off;
            // the lane's pass bits in one mask (bit EPV * j + q), then one
            // iteration per candidate: its value is read back from the stage,
            // which this warp releases only afterwards
            constexpr int NW = (VPL * EPV + 31) / 32;
            uint32_t mw[NW];
    #pragma unroll
            for (int wd = 0; wd < NW; ++wd) mw[wd] = 0;
    #pragma unroll
            for (int j = 0; j < VPL; ++j) mw[(j * EPV) / 32] |= msk[j] << ((j * EPV) % 32);
            const raw_t *selem = reinterpret_cast<const raw_t *>(svec);
    #pragma unroll
            for (int wd = 0; wd < NW; ++wd) {
                uint32_t bits = mw[wd];
                while (bits) {
                    const int e = wd * 32 + __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int epos = (vbase + (e / EPV) * kGroupWarps * 32) * EPV + (e % EPV);
                    if (slot < cap) seg[slot] = make_uint2(static_cast<uint32_t>(selem[epos]),
                                                           static_cast<uint32_t>(colbase + epos));
                    ++slot;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.empty[s]);  // release: this warp's reads of the stage are done
        }
    #ifdef GBTOPK_TRACE
        t_busy += clock64() - t_mark;
        if (threadIdx.x == 32 && kTraceBase + blockIdx.x < kTraceBlocks) {
            g_trace[kTraceBase + blockIdx.x][8] = t_wait;
            g_trace[kTraceBase + blockIdx.x][9] = t_busy;
            g_trace[kTraceBase + blockIdx.x][10] = n_items;
            g_trace[kTraceBase + blockIdx.x][11] = clock64();
        }
    #endif
    }
    // every warp is done with the ring: if a wait gave up, the finalize
    // kernel recomputes every row of this call, and the latest copy into
    // each stage must land before the block leaves (bounded wait; its phase
    // is the stage's latest)
    __syncthreads();
    if (threadIdx.x == 0 && c.abort_flag) {
        reinterpret_cast<volatile uint32_t *>(p.ws)[1] = 1u;
        const int64_t issued = c.bcast[0];
        for (int64_t i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
            if (!mbar_wait(&c.full[i % kStages], static_cast<uint32_t>((i / kStages) & 1)))
                atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusCopyLost);
    }
    GBTOPK_TRACE_POINT(6, 0);
    GBTOPK_TRACE_ANCHOR();
}


// Candidate j of a split row's concatenated chunk segments -> its address
// (the finalize's passes over segments left in L2).
struct SegMap {
    const uint2 *segs;
    const uint32_t *choff;  // first candidate number of each chunk
    int nch;
    uint32_t cap;
    // `ch` is a cursor the caller keeps: each thread visits increasing j
    __device__ __forceinline__ const uint2 *at(uint32_t j, int &ch) const {
        while (ch + 1 < nch && choff[ch + 1] <= j) ++ch;
        return segs + static_cast<int64_t>(ch) * cap + (j - choff[ch]);
    }
};

constexpr uint32_t kPadColumn = 0xFFFFFFFFu;  // marks a gather padding slot

// Coarse bin holding the r-th largest of the candidates counted in
// hist[kCoarseBins] (shared memory), found by warp 0 alone: c.bcast[2] =
// the bin, c.bcast[3] = the count above it, c.bcast[4] = its count.
// Requires 1 <= r <= the total count.  The caller syncs the block after it.
__device__ __forceinline__ void coarse_select(const uint32_t *hist, uint32_t r, Ctrl &c,
                                              uint32_t *fill = nullptr) {
    static_assert(kCoarseBins == 256, "eight bins per lane");
    if (threadIdx.x >= 32) return;
    const uint32_t lane = lane_id();
    // bins 255 - 8 lane - j, from the top (two vector loads; hist is 16-byte aligned)
    const uint4 lo = reinterpret_cast<const uint4 *>(hist)[62 - 2 * lane];
    const uint4 hi = reinterpret_cast<const uint4 *>(hist)[63 - 2 * lane];
    const uint32_t cnts[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += cnts[j];
    uint32_t incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= static_cast<uint32_t>(off)) incl += y;
    }
    const uint32_t excl = incl - s;
    if (fill) {  // fill[b] = the count of the bins above b
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            fill[255 - 8 * lane - j] = acc;
            acc += cnts[j];
        }
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, excl < r && r <= incl);
    if (bal != 0u && static_cast<int>(lane) == __ffs(bal) - 1) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (acc + cnts[j] >= r) {
                c.bcast[2] = 255u - 8u * lane - static_cast<uint32_t>(j);
                c.bcast[3] = acc;
                c.bcast[4] = cnts[j];
                break;
            }
            acc += cnts[j];
        }
    }
}

// Index of this thread among the threads of the block with `flag` set (in
// thread order), and their count.  All threads; uses c.scan; ends with a
// barrier (c.scan free again).
__device__ __forceinline__ uint32_t block_flag_index(bool flag, Ctrl &c, uint32_t &count) {
    const uint32_t warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const uint32_t m = __ballot_sync(0xffffffffu, flag);
    if (lane_id() == 0) c.scan[warp] = __popc(m);
    __syncthreads();
    uint32_t before = 0, tot = 0;
    for (uint32_t w = 0; w < nw; ++w) {
        const uint32_t v = c.scan[w];
        before += w < warp ? v : 0u;
        tot += v;
    }
    count = tot;
    const uint32_t idx = before + __popc(m & lanemask_lt());
    __syncthreads();
    return idx;
}

// Radix select among one value per thread (`live` threads): the r-th
// largest of the live values v (1 <= r <= live count), digit by digit over
// 8-bit digits from the highest bit at which the live values differ (one
// block AND/OR reduction finds it; equal values need no round).  Returns the
// value and, in gt, how many live values exceed it.  All threads; uses
// c.rhist, c.key_min, c.key_max.
__device__ __forceinline__ uint32_t block_select_one(bool live, uint32_t v, uint32_t r, Ctrl &c, uint32_t &gt) {
    if (threadIdx.x == 0) {
        c.key_min = 0xFFFFFFFFu;  // AND of the live values
        c.key_max = 0;            // OR of the live values
    }
    __syncthreads();
    const uint32_t a = __reduce_and_sync(0xffffffffu, live ? v : 0xFFFFFFFFu);
    const uint32_t o = __reduce_or_sync(0xffffffffu, live ? v : 0u);
    if (lane_id() == 0) {
        atomicAnd(&c.key_min, a);
        atomicOr(&c.key_max, o);
    }
    __syncthreads();
    const uint32_t kand = c.key_min, diff = kand ^ c.key_max;
    if (diff == 0u) {  // every live value is the same
        gt = 0;
        return kand;
    }
    const int hb = 31 - __clz(diff);           // highest differing bit
    uint32_t pmask = hb == 31 ? 0u : ~((2u << hb) - 1u);
    uint32_t prefix = kand & pmask, rem = r;
    for (int top = hb + 1; top > 0; top -= 8) {  // digits [top - 8, top), the last one clipped at bit 0
        const int shift = top > 8 ? top - 8 : 0;
        if (threadIdx.x < 256) c.rhist[threadIdx.x] = 0;
        __syncthreads();
        if (live && (v & pmask) == prefix) atomicAdd(&c.rhist[(v >> shift) & 255u], 1u);
        __syncthreads();
        coarse_select(c.rhist, rem, c);
        __syncthreads();
        const uint32_t dmask = (top >= 32 ? 0xFFFFFFFFu : ((1u << top) - 1u)) & ~((1u << shift) - 1u);
        prefix |= (c.bcast[2] << shift) & dmask;
        pmask |= dmask;
        rem -= c.bcast[3];
        __syncthreads();
    }
    gt = r - rem;
    return prefix;
}

// The best `need` of the bsize (<= NT) members of blist, by key descending
// and then by the tie mode's column order (any order for tie mode 0), into
// sel[above, above + need) in no particular order: one member per thread,
// the need-th key by block_select_one, then among the members equal to it
// either the first in list order (tie mode 0) or the ones whose tie_key is
// at most the (need - gt)-th smallest (a second select over the columns).
template <int NT, class KeyOf>
__device__ void select_members(const uint2 *blist, uint32_t bsize, uint32_t need, uint32_t above, int tie,
                               uint2 *sel, Ctrl &c, KeyOf key_of) {
    const uint32_t tid = threadIdx.x;
    const bool live = tid < bsize;
    const uint2 me = live ? blist[tid] : make_uint2(0u, 0u);
    const uint32_t mk = live ? key_of(me.x) : 0u;
    uint32_t gt;
    const uint32_t t = block_select_one(live, mk, need, c, gt);
    const uint32_t need_ties = need - gt;
    const bool eq = live && mk == t;
    bool take_eq;
    if (tie == 0) {  // (tie is block-uniform; every thread takes part in the index)
        uint32_t neq;
        const uint32_t ei = block_flag_index(eq, c, neq);
        take_eq = eq && ei < need_ties;
    } else {
        // the (need_ties)-th largest complement of tie_key = the columns to keep
        uint32_t g2;
        const uint32_t cm = ~tie_key(me.y, tie);
        const uint32_t ct = block_select_one(eq, cm, need_ties, c, g2);
        take_eq = eq && cm >= ct;
    }
    const bool take = (live && mk > t) || take_eq;
    uint32_t ntake;
    const uint32_t slot = block_flag_index(take, c, ntake);
    if (take) sel[above + slot] = me;
    __syncthreads();
}

// Completes sel[above, above + need) with the best `need` of the bsize
// members of the boundary bin (blist), ranked by (key desc, column asc).
template <int DT, int NT>
__device__ bool rank_boundary(const uint2 *blist, uint32_t bsize, uint32_t need, uint32_t above, int tie,
                              uint2 *sel, Ctrl &c) {
    if (bsize <= static_cast<uint32_t>(kRankAllMax)) {
        rank_all<DT>(const_cast<uint2 *>(blist), bsize, need, above, tie, sel);
    } else if (bsize <= static_cast<uint32_t>(NT)) {
        select_members<NT>(blist, bsize, need, above, tie, sel, c, [](uint32_t raw) { return Elem<DT>::key(raw); });
    } else {
        constexpr int KB = Elem<DT>::kKeyBits;
        const PairSrc<DT> bs{blist};
        uint32_t t, gt;
        block_select<KB, KB / 8>(bs, RankByKey{}, bsize, need, c.rhist, c, t, gt);
        const uint32_t need_ties = need - gt;
        uint32_t col_max = 0xFFFFFFFFu;
        if (tie) {
            uint32_t kk, g2;
            block_select<32, 4>(bs, RankTieColumn{t, tie}, bsize, need_ties, c.rhist, c, kk, g2);
            col_max = ~kk;
        }
        collect<DT>(bs, bsize, t, gt, need_ties, tie, col_max, sel, above, c);
    }
    return true;
}

// Where a split row's finalize keeps its data in shared memory: the kBins
// counters (the selection aliases them once they are consumed), the
// boundary-bin list, one offset per chunk, the gathered candidates, and the
// sorted-output scratch (which may reuse the list, offsets and candidates:
// they are dead once the row is selected).
struct FinalRegion {
    uint32_t *fill;       // kCoarseBins slot counters of the classification pass
    uint32_t *hist;
    uint2 *sel;
    uint2 *blist;
    uint32_t bcap;        // boundary-bin members blist holds
    uint32_t *choff;
    uint2 *cand;
    uint32_t gather_cap;  // candidates cand holds
    uint8_t *scratch;     // det_scratch_bytes(sel_cap)
};

// Exact top-k of split row `row` (n valid columns from col0, nch chunks)
// from the candidates its chunks left in the workspace.  The k-th key is
// located by a window search over the candidates' keys: first kCoarseBins
// coarse bins above the guess t_lo (coarse_bin; the row's counters from the
// workspace when the chunk kernel counted them (ws_hist), else one pass
// over the candidates), then, while the window holding the k-th key has more
// members than the boundary list holds, 8-bit sub-bins of that window.  One
// counted pass then writes every candidate above the window (to its output
// slot, or to the selection when the output is sorted) and lists the
// window's members, which are ranked exactly.  The candidates are gathered
// into shared memory by one bulk copy per chunk (each segment padded to an
// even count so every copy starts on a 16-byte boundary; the padding slot is
// marked with column kPadColumn), or read straight from L2 when they do not
// fit.  Falls back to an exact radix select over the row in global memory
// when a segment overflowed, the guess was too high (fewer than k
// candidates) or more than the list holds share the k-th key.  `bar` is an
// initialised barrier whose next phase has parity `parity`.  The next grid
// on the stream is released (programmatic dependent launch) once the
// selection is known.  All NT threads call it.
template <int DT, int NT>
__device__ void finalize_row(const Params &p, int64_t row, int64_t n, int64_t col0, int64_t nch,
                             const FinalRegion &fr, unsigned long long *bar, uint32_t parity, bool ws_hist,
                             bool recompute, Ctrl &c, int64_t trace_idx) {
    (void)trace_idx;  // the trace row of this block (GBTOPK_TRACE builds)
    using raw_t = typename Elem<DT>::raw_t;
    static_assert(NT >= kCoarseBins, "one coarse bin per thread");
    const int k = p.k;
    const bool sorted = sorted_output(p.deterministic);
    const int tie = tie_mode(p.deterministic);
    const int tid = threadIdx.x;
    const raw_t *xrow = static_cast<const raw_t *>(p.x) + row * p.row_stride + col0;
    // the row's guess, chunk counts and coarse counters: independent L2 loads, all in flight at once
    const uint2 info = __ldcg(reinterpret_cast<const uint2 *>(row_info(p, row)));
    const uint32_t my = tid < nch ? __ldcg(row_counts(p, row) + tid) : 0u;
    const uint32_t hcount = (ws_hist && tid < kCoarseBins) ? __ldcg(row_hist(p, row) + tid) : 0u;
    const uint32_t t_lo = info.x;
    const int coarse_shift = static_cast<int>(info.y);
    const uint32_t cap = static_cast<uint32_t>(chunk_seg_cap(n, k, p.plan.chunk));
    const uint2 *segs = row_segs(p, row);
    if (tid < kCoarseBins) c.rhist[tid] = hcount;
    if (tid == 0) {
        c.bcast[5] = 0;      // a chunk overflowed its segment
        c.cand_count = 0;    // chunks with an odd count
        c.sel_count = 0;
        c.b_count = 0;
    }

    // chunk counts -> padded offsets (nch <= NT, checked on the host)
    const bool over = my > cap;
    const uint32_t cnt = over ? 0u : my;
    const uint32_t padded = (cnt + 1u) & ~1u;
    __syncthreads();
    {
        const uint32_t ov = __ballot_sync(0xffffffffu, over), od = __ballot_sync(0xffffffffu, (cnt & 1u) != 0u);
        if (lane_id() == 0) {
            if (ov) atomicOr(&c.bcast[5], 1u);
            if (od) atomicAdd(&c.cand_count, static_cast<uint32_t>(__popc(od)));
        }
    }
    uint32_t total_p;
    const uint32_t poff = block_excl_scan(padded, c, total_p);  // its barriers publish the flags
    const uint32_t total = total_p - c.cand_count;
    bool fallback = recompute || c.bcast[5] != 0 || total < static_cast<uint32_t>(k);
    const bool in_smem = total_p <= fr.gather_cap;
    const bool gathered = !fallback && in_smem;  // block-uniform
    bool copy_ok = true;
    // the coarse window from the workspace counters needs no candidate: on
    // the gathered path warp 0 finds it while the copies are in flight
    const bool window_early = gathered && ws_hist;
    if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 8, -1);
    if (gathered) {
        // ---- gather the segments into shared memory (one bulk copy per chunk)
        if (tid == 0) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                         "r"(total_p * 8u)
                         : "memory");
        }
        __syncthreads();
        if (tid < nch && padded > 0) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(fr.cand + poff)),
                "l"(segs + static_cast<int64_t>(tid) * cap), "r"(padded * 8u), "r"(smem_u32(bar))
                : "memory");
        }
        if (window_early) coarse_select(c.rhist, static_cast<uint32_t>(k), c);  // (published by wait_bar's barrier)
        copy_ok = wait_bar(p.ws, c, bar, parity, p.wait_polls);
        if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 9, -1);
        if (copy_ok) {
            if (tid < nch && (cnt & 1u)) fr.cand[poff + cnt].y = kPadColumn;
            __syncthreads();
        } else {
            fallback = true;
        }
    } else if (!fallback) {
        // ---- the L2 passes need unpadded offsets
        uint32_t tot2;
        const uint32_t base = block_excl_scan(cnt, c, tot2);
        if (tid < nch) fr.choff[tid] = base;
        __syncthreads();
    }
    // visits every candidate once, in the same order on every call:
    // f(live, pair); every thread makes the same number of calls
    const SegMap map{segs, fr.choff, static_cast<int>(nch), cap};
    auto for_each_cand = [&](auto &&f) {
        if (in_smem) {
            constexpr int GS = 4;  // independent candidates per thread per step (latency overlap)
            for (uint32_t i0 = 0; i0 < total_p; i0 += GS * NT) {
                uint2 v[GS];
#pragma unroll
                for (int u = 0; u < GS; ++u) {
                    const uint32_t i = i0 + u * NT + tid;
                    v[u] = i < total_p ? fr.cand[i] : make_uint2(0u, kPadColumn);
                }
#pragma unroll
                for (int u = 0; u < GS; ++u) f(v[u].y != kPadColumn, v[u]);
            }
        } else {
            constexpr int GB = 4;  // candidates in flight per thread
            int cur = 0;
            for (uint32_t j0 = 0; j0 < total; j0 += GB * NT) {
                uint2 v[GB];
#pragma unroll
                for (int u = 0; u < GB; ++u) {
                    const uint32_t j = j0 + u * NT + tid;
                    v[u] = j < total ? __ldcg(map.at(j, cur)) : make_uint2(0u, kPadColumn);
                }
#pragma unroll
                for (int u = 0; u < GB; ++u) f(j0 + u * NT + tid < total, v[u]);
            }
        }
    };
    uint32_t above = 0, bsize = 0;
    if (!fallback) {
        if (!ws_hist) {
            for_each_cand([&](bool live, uint2 v) {
                if (live) atomicAdd(&c.rhist[coarse_bin(Elem<DT>::key(v.x), t_lo, coarse_shift)], 1u);
            });
            __syncthreads();
        }
        // ---- the window [w_lo, w_lo + 2^wbits) holding the k-th key, `above`
        // candidates above it (wbits 32: open above)
        if (!window_early) {
            coarse_select(c.rhist, static_cast<uint32_t>(k), c);
            __syncthreads();
        }
        const int s0 = coarse_shift;
        uint32_t b = c.bcast[2];
        above = c.bcast[3];
        bsize = c.bcast[4];
        uint32_t w_lo = t_lo + (b << s0);
        int wbits = b == static_cast<uint32_t>(kCoarseBins - 1) ? 32 : s0;
        while (bsize > fr.bcap && wbits > 0) {  // block-uniform: narrow the window by 8 bits
            const int sub = wbits > 8 ? wbits - 8 : 0;
            if (tid < kCoarseBins) c.rhist[tid] = 0;
            __syncthreads();
            const uint32_t wl = w_lo;
            const uint64_t wspan = uint64_t{1} << wbits;
            for_each_cand([&](bool live, uint2 v) {
                const uint32_t key = Elem<DT>::key(v.x);
                if (live && key >= wl && static_cast<uint64_t>(key - wl) < wspan)
                    atomicAdd(&c.rhist[(key - wl) >> sub], 1u);
            });
            __syncthreads();
            coarse_select(c.rhist, static_cast<uint32_t>(k) - above, c);
            __syncthreads();
            b = c.bcast[2];
            above += c.bcast[3];
            bsize = c.bcast[4];
            w_lo += b << sub;
            wbits = sub;
        }
        if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 13, -1);
        if (bsize > fr.bcap) fallback = true;  // block-uniform: more ties at the k-th key than the list holds
        if (!fallback) {
            // ---- candidates above the window to sel, its members to blist:
            // count, one block scan, write (no per-candidate atomics)
            const uint32_t wl = w_lo;
            const uint64_t wspan = uint64_t{1} << wbits;
            auto classify = [&](uint2 v, bool &hi, bool &eq) {
                const uint32_t key = Elem<DT>::key(v.x);
                const bool in = v.y != kPadColumn && key >= wl;
                const bool up = static_cast<uint64_t>(key - wl) >= wspan;
                hi = in && up;
                eq = in && !up;
            };
            constexpr int RC = 32;  // candidates per thread whose marks fit in one word
            if (in_smem && total_p <= static_cast<uint32_t>(RC * NT)) {
                // the gathered candidates stay in shared memory: mark, then
                // revisit only the marked ones
                const int nu = static_cast<int>((total_p + NT - 1) / NT);  // (block-uniform)
                uint32_t hm = 0, em = 0;
#pragma unroll 8
                for (int u = 0; u < nu; ++u) {
                    const uint32_t i = u * NT + tid;
                    if (i < total_p) {
                        bool hi, eq;
                        classify(fr.cand[i], hi, eq);
                        hm |= static_cast<uint32_t>(hi) << u;
                        em |= static_cast<uint32_t>(eq) << u;
                    }
                }
                if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 19, -1);
                uint32_t ptot;
                const uint32_t pre = block_excl_scan((static_cast<uint32_t>(__popc(hm)) << 16) | __popc(em), c, ptot);
                if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 20, -1);
                uint32_t hs = pre >> 16, es = pre & 0xFFFFu;
                while (hm) {
                    const int u = __ffs(hm) - 1;
                    hm &= hm - 1;
                    fr.sel[hs++] = fr.cand[u * NT + tid];
                }
                while (em) {
                    const int u = __ffs(em) - 1;
                    em &= em - 1;
                    fr.blist[es++] = fr.cand[u * NT + tid];
                }
                if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 21, -1);
            } else {
                uint32_t nhi = 0, neq = 0;
                for_each_cand([&](bool live, uint2 v) {
                    bool hi, eq;
                    classify(v, hi, eq);
                    nhi += (live && hi) ? 1u : 0u;
                    neq += (live && eq) ? 1u : 0u;
                });
                uint32_t ptot;
                const uint32_t pre = block_excl_scan((nhi << 16) | neq, c, ptot);
                uint32_t hs = pre >> 16, es = pre & 0xFFFFu;
                for_each_cand([&](bool live, uint2 v) {
                    bool hi, eq;
                    classify(v, hi, eq);
                    if (live && hi) fr.sel[hs++] = v;
                    if (live && eq) fr.blist[es++] = v;
                });
            }
            __syncthreads();
            if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 14, -1);
            if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 5, static_cast<int64_t>(clock64()));
            rank_boundary<DT, NT>(fr.blist, bsize, static_cast<uint32_t>(k) - above, above, tie, fr.sel, c);
        }
    }
    // the exact select uses only the selection and the control block, never
    // the gather region a timed-out copy may still be writing
    if (fallback) exact_select<DT>(GlobalSrc<DT>{xrow}, n, k, tie, fr.sel, c.rhist, c);
    if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 10, -1);
    if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 6, static_cast<int64_t>(clock64()));
    if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 11, (fallback ? 1 : 0) | (in_smem ? 2 : 0) | (static_cast<int64_t>(total) << 8));
    // the next call's first kernel may launch now (it waits for this grid
    // to complete before reading anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 15, -1);
    bool scratch_ok = true;
    if (!copy_ok) {  // the sorted output's scratch overlaps the gather region
        if (tid == 0) {
            const bool landed = mbar_wait(bar, parity);
            c.bcast[7] = landed ? 1u : 0u;
            if (!landed) atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusCopyLost);
        }
        __syncthreads();
        scratch_ok = c.bcast[7] != 0;
    }
    if (sorted && scratch_ok) {
        __syncthreads();
        emit_sorted<DT, NT>(p, row, fr.sel, k, fr.scratch, c, trace_idx);
    } else {
        emit<DT>(p, row, fr.sel, k);  // the selected set, unordered if the scratch was unusable
    }
    if (tid == 0) GBTOPK_TRACE_SET(trace_idx, 12, -1);
}

// Finalize kernel (split plans of the three-kernel path): one block per
// split row, after the stream kernel has filtered every chunk; the row is
// selected by finalize_row in this block's shared memory.
template <int DT>
__global__ void __launch_bounds__(kFinalThreads) final_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem);
    FinalRegion fr;
    fr.hist = reinterpret_cast<uint32_t *>(smem + kCtrlBytes);
    fr.sel = reinterpret_cast<uint2 *>(smem + kCtrlBytes);  // aliases hist
    fr.blist = reinterpret_cast<uint2 *>(smem + kCtrlBytes + p.plan.final_sel_bytes);
    fr.bcap = kFinalBCap;
    fr.choff = reinterpret_cast<uint32_t *>(fr.blist + kFinalBCap);
    fr.fill = fr.choff + kFinalThreads;
    fr.cand = reinterpret_cast<uint2 *>(fr.fill + kCoarseBins);  // gathered candidates
    fr.gather_cap = static_cast<uint32_t>(
        (p.plan.final_smem - (kCtrlBytes + p.plan.final_sel_bytes + static_cast<size_t>(kFinalBCap) * 8 +
                              4 * static_cast<size_t>(kFinalThreads) + 4 * static_cast<size_t>(kCoarseBins))) /
        sizeof(uint2));
    fr.scratch = reinterpret_cast<uint8_t *>(fr.cand);
    const int64_t row = p.row0 + blockIdx.x;
    constexpr int kTraceBase = kTraceFinal;
    (void)kTraceBase;
    int64_t n, col0;
    row_window(p, row, n, col0);
    const int64_t nch = split_chunks(p, n);
    if (nch == 0) return;
    if (threadIdx.x == 0) mbar_init(&c.bar);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    GBTOPK_TRACE_POINT(0, 0);
    // a stream block that gave up left some chunks unfiltered: recompute
    const bool aborted = __ldcg(reinterpret_cast<const uint32_t *>(p.ws) + 1) != 0u;
    finalize_row<DT, kFinalThreads>(p, row, n, col0, nch, fr, &c.bar, 0, false, aborted, c,
                                    kTraceFinal + blockIdx.x);
    GBTOPK_TRACE_POINT(6, 0);
    GBTOPK_TRACE_ANCHOR();
}

// Chunk kernel (split rows of plans with top_k <= kPairSortMax): one block
// per (row, chunk) slot of the launch, chunk j of a row covering its valid
// columns [j * chunk, (j + 1) * chunk); slots past a row's chunk count exit
// at once.  Each block stages its chunk by one bulk copy (issued before it
// waits for the row kernel, whose blocks have all passed their own wait for
// the stream's preceding grid, so the inputs are final), takes the row's
// guess t_lo once the row kernel has completed, keeps the chunk's elements
// >= t_lo (pass bits from one sweep over the stage, one block scan for the
// output slots, values read back from the stage) in the chunk's segment of
// the workspace and stores the chunk's count.  It then takes a ticket from
// the row's counter (cleared by the row kernel): the block that completes
// the row selects it exactly in its own shared memory (finalize_row), the
// stage being free by then.  No block ever waits for another.
template <int DT>
__global__ void __launch_bounds__(kThreads, 3) chunk_kernel(const __grid_constant__ Params p) {
    using raw_t = typename Elem<DT>::raw_t;
    constexpr int es = Elem<DT>::kBytes;
    constexpr int EPV = 16 / es;
    constexpr int VPT = kFusedStageBytes / 16 / kThreads + 1;  // stage vectors per thread
    constexpr int NW = (VPT * EPV + 31) / 32;                   // pass-bit words per thread
    static_assert(32 % EPV == 0, "a vector's pass bits never straddle two words");
    static_assert(kThreads == kCoarseBins, "one coarse bin per thread");
    static_assert(kBins * 4 + 12 * kPairSortMax <= kFusedOffSel, "sorted-output scratch below the selection");
    extern __shared__ __align__(128) uint8_t smem[];
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem);
    uint8_t *stage = smem + kCtrlBytes;
    const int tid = threadIdx.x;
    constexpr int kTraceBase = kTraceChunk;
    (void)kTraceBase;
    GBTOPK_TRACE_POINT(0, 0);
    // chunk-major slots (block b: chunk b / rows of row b % rows), so the
    // blocks of every row's first chunks, which always hold data, launch first
    const int64_t row = p.row0 + static_cast<int64_t>(blockIdx.x) % p.rows;
    const int64_t ch = static_cast<int64_t>(blockIdx.x) / p.rows;
    int64_t n, col0;
    row_window(p, row, n, col0);
    const int64_t nch = split_chunks(p, n);
    if (ch >= nch) return;
    const int64_t CH = p.plan.chunk;
    const int64_t c0 = ch * CH;
    const int len = static_cast<int>((n - c0) < CH ? (n - c0) : CH);
    const raw_t *xrow = static_cast<const raw_t *>(p.x) + row * p.row_stride + col0;
    const Span sp = span_of<DT>(xrow + c0, len);
    if (tid == 0) {
        mbar_init(&c.bar);
        bulk_load(stage, sp.a0, sp.bytes, &c.bar);
    }
    // the row kernel's guess, cleared ticket and cleared histogram
    asm volatile("griddepcontrol.wait;" ::: "memory");
    GBTOPK_TRACE_POINT(1, 0);
    uint32_t *info = row_info(p, row);
    const uint2 guess = __ldcg(reinterpret_cast<const uint2 *>(info));  // t_lo, bin shift
    if (tid == 0) c.sel_count = 0;
    c.rhist[tid] = 0;  // the chunk's coarse candidate histogram (kThreads == kCoarseBins)
    const bool ok = wait_bar(p.ws, c, &c.bar, 0, p.wait_polls);
    GBTOPK_TRACE_POINT(2, 0);
    if (ok) {
        const int nvec = ((sp.off + len) * es + 15) >> 4;
        const uint4 *svec = reinterpret_cast<const uint4 *>(stage);
        const PassTest<DT> pass(guess.x);
        uint32_t mw[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) mw[w] = 0;
        uint32_t cnt = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + j * kThreads;
            uint32_t b = 0;
            if (v < nvec) {
                b = pass.mask(svec[v]);
                if (v == 0 || v >= nvec - 1) b &= valid_lanes<EPV>(v, nvec, sp.off, len);
            }
            mw[(j * EPV) / 32] |= b << ((j * EPV) % 32);
            cnt += __popc(b);
        }
        // slots: one shared atomic per warp, lanes in order within the warp
        const uint32_t lane = lane_id();
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= static_cast<uint32_t>(o)) incl += y;
        }
        const uint32_t wtotal = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t base = 0;
        if (lane == 0 && wtotal != 0u) base = atomicAdd(&c.sel_count, wtotal);
        // the warp's candidates in rounds: each lane with candidates left
        // writes its next one, a round's slots consecutive across the lanes
        // (coalesced stores)
        uint32_t wslot = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t lt = lanemask_lt();
        const uint32_t cap = static_cast<uint32_t>(chunk_seg_cap(n, p.k, p.plan.chunk));
        uint2 *seg = row_segs(p, row) + ch * cap;
        const int shift = static_cast<int>(guess.y);
        const raw_t *selem = reinterpret_cast<const raw_t *>(stage);
        const uint32_t colbase = static_cast<uint32_t>(c0 - sp.off);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            uint32_t bits = mw[w];
            while (__any_sync(0xffffffffu, bits != 0u)) {
                const bool has = bits != 0u;
                const uint32_t m = __ballot_sync(0xffffffffu, has);
                if (has) {
                    const int e = w * 32 + __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int epos = (tid + (e / EPV) * kThreads) * EPV + (e % EPV);
                    const uint32_t raw = static_cast<uint32_t>(selem[epos]);
                    const uint32_t slot = wslot + __popc(m & lt);
                    if (slot < cap) seg[slot] = make_uint2(raw, colbase + static_cast<uint32_t>(epos));
                    atomicAdd(&c.rhist[coarse_bin(Elem<DT>::key(raw), guess.x, shift)], 1u);
                }
                wslot += __popc(m);
            }
        }
    }
    GBTOPK_TRACE_POINT(3, 0);
    // the chunk's coarse histogram into the row's (one add per nonempty
    // bin), then the ticket: the barriers and thread 0's acquire-release
    // atomic order every candidate, count and add of the block before it
    __syncthreads();
    GBTOPK_TRACE_POINT(16, 0);
    if (ok && c.rhist[tid] != 0u) atomicAdd(row_hist(p, row) + tid, c.rhist[tid]);
    __syncthreads();
    GBTOPK_TRACE_POINT(17, 0);
    if (tid == 0) {
        row_counts(p, row)[ch] = ok ? c.sel_count : 0xFFFFFFFFu;  // an unread chunk: the row falls back
        GBTOPK_TRACE_POINT(18, 0);
        // one acquire-release atomic: releases this block's candidates, count
        // and histogram adds (ordered before it by the barriers above), and
        // acquires every earlier block's for the block that completes the row
        uint32_t done;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(done) : "l"(info + 2) : "memory");
        const bool is_last = done == static_cast<uint32_t>(nch - 1);
        c.bcast[6] = is_last ? 1u : 0u;
    }
    __syncthreads();
    const bool last = c.bcast[6] != 0;
    GBTOPK_TRACE_POINT(4, 0);
    GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | (last ? 1u : 0u) |
                              (static_cast<unsigned long long>(ch) << 40));
    bool stage_ok = ok;
    if (!ok) {  // the stage copy may still land: wait (bounded) before the stage is reused or left
        if (tid == 0) {
            const bool landed = mbar_wait(&c.bar, 0);
            c.bcast[7] = landed ? 1u : 0u;
            if (!landed) atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusCopyLost);
        }
        __syncthreads();
        stage_ok = c.bcast[7] != 0;
    }
    if (!last) {
        GBTOPK_TRACE_ANCHOR();
        return;
    }
    if (!stage_ok) return;  // the row's outputs stay unwritten; the status word says so
    FinalRegion fr;
    fr.hist = nullptr;
    fr.sel = reinterpret_cast<uint2 *>(stage + kFusedOffSel);
    fr.blist = reinterpret_cast<uint2 *>(stage);
    fr.bcap = kFusedBCap;
    fr.choff = reinterpret_cast<uint32_t *>(stage + kFusedOffChOff);
    fr.fill = reinterpret_cast<uint32_t *>(stage + kFusedOffFill);
    fr.cand = reinterpret_cast<uint2 *>(stage + kFusedOffCand);
    fr.gather_cap = kFusedGatherCap;
    fr.scratch = stage;  // det_scratch_bytes(2048) = 40 KB, below the selection
    finalize_row<DT, kThreads>(p, row, n, col0, nch, fr, &c.bar, 1, true, false, c, kTraceChunk + blockIdx.x);
    GBTOPK_TRACE_ANCHOR();
}

// ---------------------------------------------------------------- small rows

// Small-row kernel (widths up to 32 * NE <= 2048 columns, calls without the
// sorted output order): one warp per row, no block barrier.  Lane l holds
// columns l, l + 32, ..., as keys in registers.  The k-th largest key t
// comes from a radix select over 8-bit digits with a warp-private 256-bin
// shared histogram (two rounds for 16-bit keys, four for fp32).  The keys
// above t and k - #(keys > t) keys equal to t (the first in column order,
// or the last with the largest-columns tie mode) are then written in column
// order, each warp-wide slot from two ballots per register.
template <int DT, int NE>
__global__ void __launch_bounds__(128) small_kernel(const __grid_constant__ Params p) {
    using raw_t = typename Elem<DT>::raw_t;
    constexpr int KB = Elem<DT>::kKeyBits;
    const uint32_t lane = lane_id();
    __shared__ uint32_t small_hist[4 * 256];  // one digit histogram per warp
    // a programmatic dependent of the stream's preceding kernel (see the
    // row kernel); the next call may launch once every row is selected
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    if (row >= p.num_rows) return;  // whole warps
    const int k = p.k;
    int64_t n, col0;
    row_window(p, row, n, col0);
    const raw_t *xrow = static_cast<const raw_t *>(p.x) + row * p.row_stride + col0;
    int32_t *out = p.out_idx + row * k;
    // the unrolled selection below stores bare column indices in out; a
    // rolled pass then applies the page-table transform and the values
    if (n <= k) {  // short and empty rows: every valid column in order, then -1
        for (int64_t j = lane; j < k; j += 32) out[j] = j < n ? static_cast<int32_t>(j) : -1;
    } else {
        uint32_t key[NE];
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int64_t c = lane + 32 * e;
            key[e] = c < n ? Elem<DT>::key(ldg_raw(xrow + c)) : 0u;
        }
        // the k-th largest key: radix select over 8-bit digits from the top,
        // one 256-bin shared histogram per warp (columns past the row hold
        // key 0, which no real value maps to, and are left out)
        uint32_t *h = small_hist + (threadIdx.x >> 5) * 256;
        uint32_t prefix = 0, pmask = 0, rem = static_cast<uint32_t>(k), bin_n = 0;
#pragma unroll 1
        for (int shift = KB - 8; shift >= 0; shift -= 8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) h[lane + 32 * i] = 0;
            __syncwarp();
#pragma unroll
            for (int e = 0; e < NE; ++e)
                if (key[e] != 0u && (key[e] & pmask) == prefix) atomicAdd(&h[(key[e] >> shift) & 255u], 1u);
            __syncwarp();
            uint32_t cnt[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cnt[j] = h[255 - 8 * lane - j];
                sum += cnt[j];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= static_cast<uint32_t>(o)) incl += y;
            }
            const uint32_t excl = incl - sum;
            const uint32_t owner = __ffs(__ballot_sync(0xffffffffu, excl < rem && rem <= incl)) - 1;
            uint32_t digit = 0, above = excl, nd = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (above + cnt[j] >= rem) {
                    digit = 255u - 8u * lane - static_cast<uint32_t>(j);
                    nd = cnt[j];
                    break;
                }
                above += cnt[j];
            }
            digit = __shfl_sync(0xffffffffu, digit, owner);
            above = __shfl_sync(0xffffffffu, above, owner);
            bin_n = __shfl_sync(0xffffffffu, nd, owner);  // after the last digit: #(keys == t)
            prefix |= digit << shift;
            pmask |= 255u << shift;
            rem -= above;
            __syncwarp();
        }
        const uint32_t t = prefix;
        const uint32_t gt = static_cast<uint32_t>(k) - rem;
        // ties taken: the first `need` in column order, or with the
        // largest-columns tie mode the last `need` (the first `skip` are passed over)
        const uint32_t need = rem;
        const uint32_t skip = tie_mode(p.deterministic) == 2 ? bin_n - need : 0u;
        const uint32_t lt = lanemask_lt();
        uint32_t hi_base = 0, tie_base = 0;
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const bool h = key[e] > t, q = key[e] == t;
            const uint32_t bh = __ballot_sync(0xffffffffu, h);
            const uint32_t bt = __ballot_sync(0xffffffffu, q);
            const uint32_t r = tie_base + __popc(bt & lt) - skip;  // wraps for passed-over ties
            const uint32_t slot = h ? hi_base + __popc(bh & lt) : gt + r;
            if (h || (q && r < need)) out[slot] = static_cast<int32_t>(lane + 32 * e);
            hi_base += __popc(bh);
            tie_base += __popc(bt);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!p.page_table && !p.idx_offset && !p.out_val) return;
    __syncwarp();  // the warp's index stores are visible to its lanes
    const RowEpi ep = row_epilogue(p, row);
#pragma unroll 1
    for (int64_t j = lane; j < k; j += 32) {
        const int32_t idx = out[j];
        if (p.out_val)
            static_cast<raw_t *>(p.out_val)[row * k + j] =
                static_cast<raw_t>(idx >= 0 ? ldg_raw(xrow + idx) : Elem<DT>::kLowest);
        if (p.page_table || p.idx_offset) {
            if (p.out_raw) p.out_raw[row * k + j] = idx;
            out[j] = out_index(p, ep, idx);
        }
    }
}

// Elem16::key of both halves of a word at once: a half whose magnitude is
// zero loses its sign bit (-0 -> +0), then the negative halves are inverted
// and the others get their top bit set.
__device__ __forceinline__ uint32_t pair_keys(uint32_t w) {
    const uint32_t nz = ((w & 0x7FFF7FFFu) + 0x7FFF7FFFu) & 0x80008000u;  // halves with a nonzero magnitude
    const uint32_t v = w & (0x7FFF7FFFu | nz);
    const uint32_t neg = prmt(v, 0u, 0xBB99u);  // 0xFFFF in each half whose sign bit is set
    return v ^ (neg | 0x80008000u);
}

// Bit 15 (31) set iff the low (high) 16-bit half of a is >= the matching
// half of T, for unsigned halves; Tlo = T & 0x7FFF7FFF.  The low 15 bits of
// each half are compared by a subtraction that cannot borrow across halves
// ((a | 0x8000) - (T & 0x7FFF) > 0), and the top bits decide where they
// differ.  Other bits of the result are meaningless.
__device__ __forceinline__ uint32_t pair_ge(uint32_t a, uint32_t T, uint32_t Tlo) {
    const uint32_t x = (a | 0x80008000u) - Tlo;
    return (a & ~T) | (~(a ^ T) & x);
}

// The digit holding the rem-th largest of the 256 counters h (shared
// memory, one warp), counting from the top, after taking sub0 off bin 0:
// the digit, the count of the bins above it and its own count.
__device__ __forceinline__ void warp_digit(const uint32_t *h, uint32_t rem, uint32_t sub0, uint32_t &digit,
                                           uint32_t &above, uint32_t &cnt) {
    const uint32_t lane = lane_id();
    // lane l owns bins 255 - 8 l down to 248 - 8 l
    const uint4 lo = reinterpret_cast<const uint4 *>(h)[62 - 2 * lane];
    const uint4 hi = reinterpret_cast<const uint4 *>(h)[63 - 2 * lane];
    uint32_t c[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};
    if (lane == 31) c[7] -= sub0;
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += c[j];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= static_cast<uint32_t>(o)) incl += y;
    }
    const uint32_t excl = incl - sum;
    const uint32_t owner = __ffs(__ballot_sync(0xffffffffu, excl < rem && rem <= incl)) - 1;
    uint32_t d = 0, a = excl, nd = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (a + c[j] >= rem) {
            d = 255u - 8u * lane - static_cast<uint32_t>(j);
            nd = c[j];
            break;
        }
        a += c[j];
    }
    digit = __shfl_sync(0xffffffffu, d, owner);
    above = __shfl_sync(0xffffffffu, a, owner);
    cnt = __shfl_sync(0xffffffffu, nd, owner);
}

// The selection of one 16-bit row of nn > k valid columns by one warp
// (small16_kernel): word w of lane l holds the keys of columns
// 2 (l + 32 w) and 2 (l + 32 w) + 1, packed (pair_keys), and key_word(w)
// returns it for the words w < nwv that hold valid columns; padding halves
// hold key 0 (the raw value 0xFFFF), whose count is taken off digit 0 of
// each histogram.  The k-th largest key t comes from two 8-bit radix rounds
// over the warp's shared histogram h.  The output lists the keys > t and
// the first need = k - #(keys > t) keys equal to t in column order (the
// last ones with the largest-columns tie mode), word by word with two
// ballots per word; when every key equal to t is taken, one packed compare
// per word (pair_ge) decides.
template <class KeyWord>
__device__ __forceinline__ void small16_select(const Params &p, int nn, int nwv, uint32_t *h, int32_t *out,
                                               const KeyWord &key_word) {
    const uint32_t lane = lane_id();
    const int k = p.k;
    const uint32_t pad = static_cast<uint32_t>(64 * nwv - nn);  // padding halves in the visited words
    // round 1: the top byte of the key
    reinterpret_cast<uint4 *>(h)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(h)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
#pragma unroll 4
    for (int w = 0; w < nwv; ++w) {
        const uint32_t kw = key_word(w);
        atomicAdd(&h[prmt(kw, 0u, 0x4441u)], 1u);
        atomicAdd(&h[kw >> 24], 1u);
    }
    __syncwarp();
    uint32_t d1, above, cnt;
    uint32_t rem = static_cast<uint32_t>(k);
    warp_digit(h, rem, pad, d1, above, cnt);
    rem -= above;
    __syncwarp();
    // round 2: the low byte, among the keys whose top byte is d1
    reinterpret_cast<uint4 *>(h)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(h)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    const uint32_t pat = d1 * 0x01000100u;
#pragma unroll 4
    for (int w = 0; w < nwv; ++w) {
        const uint32_t kw = key_word(w);
        const uint32_t x = kw ^ pat;
        if ((x & 0xFF00u) == 0u) atomicAdd(&h[kw & 0xFFu], 1u);
        if (x < 0x01000000u) atomicAdd(&h[prmt(kw, 0u, 0x4442u)], 1u);
    }
    __syncwarp();
    uint32_t d2, bin_n;
    warp_digit(h, rem, d1 == 0u ? pad : 0u, d2, above, bin_n);
    rem -= above;
    const uint32_t t = (d1 << 8) | d2;
    const uint32_t gt = static_cast<uint32_t>(k) - rem;  // keys > t
    const uint32_t need = rem;                           // keys == t to take (1 <= need <= bin_n)
    const uint32_t lt = lanemask_lt();
    const uint32_t T = t | (t << 16);
    uint32_t base = 0;
    if (need == bin_n) {  // the output is every key >= t
        const uint32_t Tlo = T & 0x7FFF7FFFu;
#pragma unroll 4
        for (int w = 0; w < nwv; ++w) {
            const uint32_t ge = pair_ge(key_word(w), T, Tlo);
            const bool p0 = (ge & 0x8000u) != 0u, p1 = (ge & 0x80000000u) != 0u;
            const uint32_t b0 = __ballot_sync(0xffffffffu, p0), b1 = __ballot_sync(0xffffffffu, p1);
            const uint32_t s0 = base + __popc(b0 & lt) + __popc(b1 & lt);
            const int32_t c = 2 * (static_cast<int32_t>(lane) + 32 * w);
            if (p0) out[s0] = c;
            if (p1) out[s0 + (p0 ? 1u : 0u)] = c + 1;
            base += __popc(b0) + __popc(b1);
        }
    } else {  // some keys equal to t are left out: ties ranked in column order
        const uint32_t skip = tie_mode(p.deterministic) == 2 ? bin_n - need : 0u;
        uint32_t tie_base = 0;
#pragma unroll 2
        for (int w = 0; w < nwv; ++w) {
            const uint32_t a = key_word(w);
            const uint32_t k0 = a & 0xFFFFu, k1 = a >> 16;
            const bool g0 = k0 > t, g1 = k1 > t, q0 = k0 == t, q1 = k1 == t;
            const uint32_t bg0 = __ballot_sync(0xffffffffu, g0), bg1 = __ballot_sync(0xffffffffu, g1);
            const uint32_t bq0 = __ballot_sync(0xffffffffu, q0), bq1 = __ballot_sync(0xffffffffu, q1);
            const uint32_t hs = base + __popc(bg0 & lt) + __popc(bg1 & lt);
            const uint32_t r0 = tie_base + __popc(bq0 & lt) + __popc(bq1 & lt) - skip;  // wraps when passed over
            const uint32_t r1 = r0 + (q0 ? 1u : 0u);
            const int32_t c = 2 * (static_cast<int32_t>(lane) + 32 * w);
            if (g0) out[hs] = c;
            if (g1) out[hs + (g0 ? 1u : 0u)] = c + 1;
            if (q0 && r0 < need) out[gt + r0] = c;
            if (q1 && r1 < need) out[gt + r1] = c + 1;
            base += __popc(bg0) + __popc(bg1);
            tie_base += __popc(bq0) + __popc(bq1);
        }
    }
}

// Small-row kernel for 16-bit rows (widths up to 64 * NW <= 2048, calls
// without the sorted order): one warp per row, no block barrier.  A row
// longer than k is staged by one bulk copy (its bytes all in flight at
// once), turned into packed keys in place and selected by small16_select;
// if the copy does not land within the first bounded wait, the keys are
// read from global memory instead (status bit 0), and the warp waits again
// (bounded) for the copy before it leaves.
template <int DT, int NW>
__global__ void __launch_bounds__(128, 7) small16_kernel(const __grid_constant__ Params p) {
    static_assert(Elem<DT>::kBytes == 2, "16-bit rows");
    using raw_t = typename Elem<DT>::raw_t;
    const uint32_t lane = lane_id();
    const uint32_t wid = threadIdx.x >> 5;
    constexpr int kStageWords = 32 * NW + 8;  // a row of 64 NW columns and the 16-byte rounding on both sides
    __shared__ __align__(16) uint32_t small_hist[4 * 256];  // one digit histogram per warp
    __shared__ __align__(16) uint32_t small_stage[4][kStageWords];
    __shared__ unsigned long long small_bar[4];
    constexpr int kTraceBase = 0;
    (void)kTraceBase;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    GBTOPK_TRACE_POINT(0, 0);
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + wid;
    if (row >= p.num_rows) return;  // whole warps
    const int k = p.k;
    int64_t n, col0;
    row_window(p, row, n, col0);
    const raw_t *xrow = static_cast<const raw_t *>(p.x) + row * p.row_stride + col0;
    int32_t *out = p.out_idx + row * k;
    if (n <= k) {  // short and empty rows: every valid column in order, then -1
        for (int64_t j = lane; j < k; j += 32) out[j] = j < n ? static_cast<int32_t>(j) : -1;
    } else {
        const int nn = static_cast<int>(n);
        const int nwv = (nn + 63) >> 6;  // words with a valid column (warp-uniform)
        const Span sp = span_of<DT>(xrow, n);
        unsigned long long *bar = &small_bar[wid];
        uint32_t *stage = small_stage[wid];
        uint32_t *h = small_hist + wid * 256;
        if (lane == 0) {
            mbar_init(bar);
            bulk_load(stage, sp.a0, sp.bytes, bar);
        }
        uint32_t landed = lane == 0 ? (mbar_wait(bar, 0, p.wait_polls) ? 1u : 0u) : 0u;
        landed = __shfl_sync(0xffffffffu, landed, 0);
        if (landed) {
            mbar_wait(bar, 0);  // completes at once: every lane sees the copied bytes
            // the packed keys, in place: word w of lane l to stage[l + 32 w]
            // (an odd first element straddles two copied words)
            const int sh = (sp.off & 1) * 16;
            const int wb = sp.off >> 1;
            for (int w = 0; w < nwv; ++w) {
                const int q = wb + static_cast<int>(lane) + 32 * w;
                uint32_t v = __funnelshift_r(stage[q], stage[q + 1], sh);
                const int c = 2 * (static_cast<int>(lane) + 32 * w);
                if (c >= nn) v |= 0xFFFFu;
                if (c + 1 >= nn) v |= 0xFFFF0000u;
                __syncwarp();  // every lane has read before any lane writes
                stage[lane + 32 * w] = pair_keys(v);
            }
            __syncwarp();
            GBTOPK_TRACE_POINT(1, 0);
            small16_select(p, nn, nwv, h, out, [&](int w) { return stage[lane + 32 * w]; });
        } else {  // the copy did not land in time: read the row from global memory
            if (lane == 0) atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusWaitTimeout);
            small16_select(p, nn, nwv, h, out, [&](int w) {
                const int c = 2 * (static_cast<int>(lane) + 32 * w);
                const uint32_t lo = c < nn ? ldg_raw(xrow + c) : 0xFFFFu;
                const uint32_t hi = c + 1 < nn ? ldg_raw(xrow + c + 1) : 0xFFFFu;
                return pair_keys(lo | (hi << 16));
            });
            if (lane == 0 && !mbar_wait(bar, 0))  // the stage must not be left with a copy in flight
                atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusCopyLost);
            __syncwarp();
        }
    }
    GBTOPK_TRACE_POINT(4, 0);
    GBTOPK_TRACE_POINT(7, static_cast<unsigned long long>(n));
    GBTOPK_TRACE_ANCHOR();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!p.page_table && !p.idx_offset && !p.out_val) return;
    __syncwarp();  // the warp's index stores are visible to its lanes
    const RowEpi ep = row_epilogue(p, row);
#pragma unroll 1
    for (int64_t j = lane; j < k; j += 32) {
        const int32_t idx = out[j];
        if (p.out_val)
            static_cast<raw_t *>(p.out_val)[row * k + j] =
                static_cast<raw_t>(idx >= 0 ? ldg_raw(xrow + idx) : Elem<DT>::kLowest);
        if (p.page_table || p.idx_offset) {
            if (p.out_raw) p.out_raw[row * k + j] = idx;
            out[j] = out_index(p, ep, idx);
        }
    }
}

template <int DT, int NW>
cudaError_t launch_small16(const Params &p, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>((p.num_rows + 3) / 4);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, small16_kernel<DT, NW>, p);
}

template <int DT, int NE>
cudaError_t launch_small(const Params &p, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>((p.num_rows + 3) / 4);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, small_kernel<DT, NE>, p);
}

// Opts kernel `kern` into `bytes` of dynamic shared memory on the current
// device when that is above the 48 KB default.  The attribute is per device
// and per kernel, so the largest opt-in so far is remembered per (device,
// kernel), under a lock shared by every host thread.
std::mutex g_smem_mutex;
std::map<std::pair<int, const void *>, size_t> g_smem_opted;

template <class K>
cudaError_t set_smem(K kern, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const std::pair<int, const void *> key(dev, reinterpret_cast<const void *>(kern));
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    const auto it = g_smem_opted.find(key);
    if (it != g_smem_opted.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    g_smem_opted[key] = bytes;
    return cudaSuccess;
}

template <int DT, int VPT>
cudaError_t launch_row(const Params &p, cudaStream_t stream) {
    const size_t bytes = sorted_output(p.deterministic) ? p.plan.row_smem_sorted : p.plan.row_smem;
    const cudaError_t e = set_smem(row_kernel<DT, VPT>, bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.rows));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, row_kernel<DT, VPT>, p);
}

// Row-kernel variant by the vectors each thread holds for a direct row.
template <int DT>
cudaError_t launch_row_any(const Params &p, cudaStream_t stream) {
    if (p.plan.split) return launch_row<DT, 0>(p, stream);
    const int64_t vec = (static_cast<int64_t>(p.plan.direct_max) * Elem<DT>::kBytes + 16 + 15) / 16;
    if (vec <= 3 * kThreads) return launch_row<DT, 3>(p, stream);
    if (vec <= 9 * kThreads) return launch_row<DT, 9>(p, stream);
    return launch_row<DT, 17>(p, stream);
}

template <int DT>
cudaError_t launch_dt(const Params &p0, cudaStream_t stream) {
    cudaError_t e;
    if (!p0.plan.split) {
        Params p = p0;
        p.row0 = 0;
        p.rows = p0.num_rows;
        if (!sorted_output(p.deterministic) && p.width <= 32 * 64) {  // one warp per row
            if constexpr (Elem<DT>::kBytes == 2) {
                if (p.width <= 64 * 8) return launch_small16<DT, 8>(p, stream);
                if (p.width <= 64 * 16) return launch_small16<DT, 16>(p, stream);
                return launch_small16<DT, 32>(p, stream);
            } else {
                if (p.width <= 32 * 16) return launch_small<DT, 16>(p, stream);
                if (p.width <= 32 * 32) return launch_small<DT, 32>(p, stream);
                return launch_small<DT, 64>(p, stream);
            }
        }
        return launch_row_any<DT>(p, stream);
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    if (p0.plan.fused) {
        // row kernel (guesses, short rows), then one chunk-kernel block per
        // (row, chunk) slot, in launches of up to block_rows rows
        if ((e = set_smem(chunk_kernel<DT>, p0.plan.fused_smem)) != cudaSuccess) return e;
        for (int64_t r0 = 0; r0 < p0.num_rows; r0 += p0.plan.block_rows) {
            Params p = p0;
            p.row0 = r0;
            p.rows = (p0.num_rows - r0) < p0.plan.block_rows ? (p0.num_rows - r0) : p0.plan.block_rows;
            if ((e = launch_row_any<DT>(p, stream)) != cudaSuccess) return e;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(p.rows * p.plan.chunks_per_row));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = p.plan.fused_smem;
            cfg.stream = stream;
            cfg.attrs = pdl;
            cfg.numAttrs = 1;
            if ((e = cudaLaunchKernelEx(&cfg, chunk_kernel<DT>, p)) != cudaSuccess) return e;
        }
        return cudaGetLastError();
    }
    if ((e = set_smem(stream_kernel<DT>, p0.plan.stream_smem)) != cudaSuccess) return e;
    if ((e = set_smem(final_kernel<DT>, p0.plan.final_smem)) != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int64_t r0 = 0; r0 < p0.num_rows; r0 += p0.plan.block_rows) {
        Params p = p0;
        p.row0 = r0;
        p.rows = (p0.num_rows - r0) < p0.plan.block_rows ? (p0.num_rows - r0) : p0.plan.block_rows;
        if ((e = launch_row_any<DT>(p, stream)) != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sms));
        cfg.blockDim = dim3(kStreamThreads);
        cfg.dynamicSmemBytes = p.plan.stream_smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, stream_kernel<DT>, p)) != cudaSuccess) return e;
        cfg.gridDim = dim3(static_cast<unsigned>(p.rows));
        cfg.blockDim = dim3(kFinalThreads);
        cfg.dynamicSmemBytes = p.plan.final_smem;
        if ((e = cudaLaunchKernelEx(&cfg, final_kernel<DT>, p)) != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

#ifdef GBTOPK_TRACE
extern "C" int gbtopk_trace_read(void *host, size_t bytes) {
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return cudaMemcpyFromSymbol(host, g_trace, bytes) == cudaSuccess ? 0 : -5;
}
#endif

cudaError_t launch_topk(int dtype, const Params &p, cudaStream_t stream) {
    switch (dtype) {
        case 0: return launch_dt<0>(p, stream);
        case 1: return launch_dt<1>(p, stream);
        case 2: return launch_dt<2>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbtopk

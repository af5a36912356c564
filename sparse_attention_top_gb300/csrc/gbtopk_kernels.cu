// Device code of gbtopk: batched variable-length exact top-K on sm_103a.
//
// One launch serves a whole ragged batch.  Block b handles chunk b % C of
// row b / C (C = chunks per row, fixed by the launch plan from the buffer
// width only, so the geometry never depends on seq_lens contents and the
// call is CUDA-graph safe; TensorRT-LLM PR #17821, run_varlen commits).
//
// Per row (valid length n, from the FlashInfer `top_k_varlen` seq_lens
// formula or from the page-table call's lengths / row_starts):
//   * n == 0            -> all -1 (zero-window rows).
//   * n <= k            -> every valid column, then -1 (short path).
//   * k < n <= chunk    -> the row is staged in shared memory by one bulk
//                          asynchronous copy and an exact radix select runs
//                          on it (8-bit digits, shared-memory histograms with
//                          warp-aggregated atomics).
//   * n > chunk         -> split: each block stages its chunk, guesses a
//                          threshold from a strided sample of the row (the
//                          self-sampling guess of TensorRT-LLM PR #17821,
//                          optionally anchored at the hint's argmax), keeps
//                          the candidates at or above it with a histogram of
//                          their keys, and publishes both to the workspace.
//                          The last block of the row (atomic ticket) finds
//                          the exact k-th key from the histogram and the
//                          candidates, and restores the workspace to zero.
//                          If the guess was too high or a buffer overflowed
//                          (count-crossing check), that block recomputes the
//                          row with the exact select from global memory, so
//                          the result never depends on the guess.
// Ranking uses order-preserving integer keys (signed zeros equal; +-inf and
// denormals exact), so no float compare depends on flush-to-zero.
#include <cstdint>

#include <cuda_runtime.h>

#include "gbtopk_internal.h"

namespace gbtopk {

#ifdef GBTOPK_TRACE
// Phase timestamps (%globaltimer, ns) of the first kTraceBlocks blocks, for
// builds compiled with -DGBTOPK_TRACE (read back by gbtopk_trace_read).
constexpr int kTraceBlocks = 1 << 16;
__device__ unsigned long long g_trace[kTraceBlocks][8];
#define GBTOPK_TRACE_POINT(slot, value)                                        \
    do {                                                                       \
        if (threadIdx.x == 0 && blockIdx.x < kTraceBlocks) {                   \
            unsigned long long t_;                                             \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));             \
            g_trace[blockIdx.x][slot] = (slot) == 7 ? (value) : t_;            \
        }                                                                      \
    } while (0)
#else
#define GBTOPK_TRACE_POINT(slot, value) \
    do {                                \
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
    static constexpr uint32_t kKeyZeroRaw = 0xFFFFFFFFu; // a raw whose key is 0
    __device__ __forceinline__ static uint32_t key(uint32_t u) {
        u = (u == 0x80000000u) ? 0u : u;
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
};

struct Elem16 {
    using raw_t = uint16_t;
    static constexpr int kBytes = 2;
    static constexpr int kKeyBits = 16;
    static constexpr uint32_t kKeyZeroRaw = 0xFFFFu;
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
    uint32_t pad[3];
    uint32_t scan[72];
    uint32_t rhist[256];     // radix-select digit histogram
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

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

// Waits for phase `parity` of the barrier; gives up after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity) {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
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

template <int DT>
struct GlobalPairSrc {  // (raw, column) pairs published by other blocks (read from L2)
    static constexpr int kBatch = 8;
    const uint2 *p;
    __device__ __forceinline__ void get(int64_t i, uint32_t &key, uint32_t &idx, uint32_t &raw) const {
        const uint2 v = __ldcg(p + i);
        raw = v.x;
        key = Elem<DT>::key(v.x);
        idx = v.y;
    }
};

struct KeyArraySrc {  // keys already mapped (the row sample)
    static constexpr int kBatch = 8;
    const uint32_t *k;
    __device__ __forceinline__ void get(int64_t i, uint32_t &key, uint32_t &idx, uint32_t &raw) const {
        key = k[i];
        idx = static_cast<uint32_t>(i);
        raw = 0;
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

struct RankTieColumn {
    uint32_t t;
    __device__ __forceinline__ bool operator()(uint32_t key, uint32_t idx, uint32_t &k) const {
        k = ~idx;
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
// items with key == t into sel[base + gt ..).  Deterministic mode keeps the
// ties whose column is <= tie_col_max (exactly need_ties of them).
template <int DT, class S>
__device__ void collect(const S &s, int64_t cnt, uint32_t t, uint32_t gt, uint32_t need_ties,
                        bool det, uint32_t tie_col_max, uint2 *sel, uint32_t base, Ctrl &c) {
    if (threadIdx.x == 0) {
        c.sel_count = 0;
        c.tie_count = 0;
    }
    __syncthreads();
    for_each_item(s, cnt, [&](bool valid, uint32_t key, uint32_t idx, uint32_t raw) {
        const bool above = valid && key > t;
        const bool tie = valid && key == t && (!det || idx <= tie_col_max);
        const uint32_t slot = warp_claim(&c.sel_count, above);
        if (above) sel[base + slot] = make_uint2(raw, idx);
        const uint32_t tslot = warp_claim(&c.tie_count, tie);
        if (tie && tslot < need_ties) sel[base + gt + tslot] = make_uint2(raw, idx);
    });
    __syncthreads();
}

// Exact top-k (n > k) of a source into sel[0..k).
template <int DT, class S>
__device__ void exact_select(const S &s, int64_t n, int k, bool det, uint2 *sel, uint32_t *hist,
                             Ctrl &c) {
    constexpr int KB = Elem<DT>::kKeyBits;
    uint32_t t, gt;
    block_select<KB, KB / 8>(s, RankByKey{}, n, static_cast<uint32_t>(k), hist, c, t, gt);
    const uint32_t need_ties = static_cast<uint32_t>(k) - gt;
    uint32_t col_max = 0xFFFFFFFFu;
    if (det) {
        uint32_t kk, g2;
        block_select<32, 4>(s, RankTieColumn{t}, n, need_ties, hist, c, kk, g2);
        col_max = ~kk;
    }
    collect<DT>(s, n, t, gt, need_ties, det, col_max, sel, 0, c);
}

// Orders sel[0..m) by (key desc, column asc) with a bitonic network over the
// next power of two; the padding sorts last.
template <int DT>
__device__ void sort_selection(uint2 *sel, int m) {
    int p2 = 1;
    while (p2 < m) p2 <<= 1;
    for (int i = m + threadIdx.x; i < p2; i += blockDim.x)
        sel[i] = make_uint2(Elem<DT>::kKeyZeroRaw, 0x7FFFFFFFu);
    __syncthreads();
    auto comp = [](uint2 v) -> unsigned long long {
        return (static_cast<unsigned long long>(Elem<DT>::key(v.x)) << 32) |
               static_cast<unsigned long long>(0xFFFFFFFFu - v.y);
    };
    for (int size = 2; size <= p2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (p2 >> 1); i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint2 a = sel[lo], b = sel[hi];
                if ((comp(a) < comp(b)) == desc) {
                    sel[lo] = b;
                    sel[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- row geometry and output

__device__ __forceinline__ void row_window(const Params &p, int64_t row, int64_t &n, int64_t &col0) {
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

template <int DT>
__device__ void emit(const Params &p, int64_t row, const uint2 *sel, int m) {
    using raw_t = typename Elem<DT>::raw_t;
    const int k = p.k;
    int64_t pt_start = 0;
    if (p.page_table) {
        if (p.pt_row_starts) pt_start = __ldg(p.pt_row_starts + row);
        else if (p.pt_start_is_row_start) pt_start = __ldg(p.row_starts + row);
    }
    int32_t *out = p.out_idx + row * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        const bool live = j < m;
        const int32_t idx = live ? static_cast<int32_t>(sel[j].y) : -1;
        if (p.page_table) {
            int32_t v = -1;
            if (idx >= 0) {
                const int64_t col = pt_start + idx / p.page_size;
                if (col >= 0 && col < p.pt_cols) {
                    const int64_t page = __ldg(p.page_table + row * p.pt_row_stride + col);
                    v = static_cast<int32_t>(static_cast<uint32_t>(
                        static_cast<uint64_t>(page * p.page_size + idx % p.page_size)));
                }
            }
            out[j] = v;
            if (p.out_raw) p.out_raw[row * k + j] = idx;
        } else {
            out[j] = idx;
        }
        if (p.out_val)
            static_cast<raw_t *>(p.out_val)[row * k + j] =
                static_cast<raw_t>(live ? sel[j].x : Elem<DT>::kLowest);
    }
}

// Stages elements [0, len) of `src` into shared memory: the 16-byte aligned
// body by one bulk asynchronous copy, the unaligned head and tail by plain
// loads.  Element e lands at stage[off + e].  Returns the body byte count
// (0: nothing to wait for).  Thread 0 issues the copy.
template <int DT>
__device__ uint32_t stage_row(const typename Elem<DT>::raw_t *src, int64_t len,
                              typename Elem<DT>::raw_t *stage, unsigned long long *bar, int &off) {
    constexpr int es = Elem<DT>::kBytes;
    const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
    off = static_cast<int>(mis / es);
    int64_t head = static_cast<int64_t>(((16u - mis) & 15u) / es);
    if (head > len) head = len;
    const uint32_t body_bytes = static_cast<uint32_t>(((len - head) * es) & ~static_cast<int64_t>(15));
    const int64_t body_end = head + body_bytes / es;
    if (threadIdx.x == 0 && body_bytes) bulk_load(stage + off + head, src + head, body_bytes, bar);
    for (int64_t e = threadIdx.x; e < head; e += blockDim.x) stage[off + e] = __ldg(src + e);
    for (int64_t e = body_end + threadIdx.x; e < len; e += blockDim.x) stage[off + e] = __ldg(src + e);
    return body_bytes;
}

// Block-uniform wait for the staged body.  On timeout the status word is
// flagged and the caller recomputes from global memory.
__device__ bool wait_stage(const Params &p, Ctrl &c, uint32_t body_bytes) {
    if (body_bytes == 0) return true;
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait(&c.bar, 0);
        c.bcast[7] = ok ? 1u : 0u;
        if (!ok) atomicOr(reinterpret_cast<uint32_t *>(p.ws), kStatusWaitTimeout);
    }
    __syncthreads();
    const bool ok = c.bcast[7] != 0;
    if (ok) mbar_wait(&c.bar, 0);  // completes at once; acquire for every thread
    __syncthreads();
    return ok;
}

__device__ void drain_stage(Ctrl &c, uint32_t body_bytes, bool waited_ok) {
    if (threadIdx.x == 0 && body_bytes && !waited_ok) mbar_wait(&c.bar, 0);
}

// ---------------------------------------------------------------- threshold guess

// From m sample keys in shared memory, the guess t_lo: the r-th largest
// sample key truncated to its top 16 bits, with r chosen so that the count
// of row elements >= t_lo falls below k only with a tiny probability
// (r = e + 6 sqrt(e) + 2, e = m k / n the expected sample count at or above
// the k-th largest).  Also the histogram scale: keys t_lo .. key_max map
// onto the lower half of kBins bins.
template <int DT>
__device__ void guess_threshold(const uint32_t *sample, int m, int64_t n, int k, uint32_t key_max,
                                Ctrl &c, uint32_t &t_lo, int &bin_shift) {
    constexpr int KB = Elem<DT>::kKeyBits;
    const double e = static_cast<double>(m) * k / static_cast<double>(n);
    uint32_t r = static_cast<uint32_t>(ceil(e + 6.0 * sqrt(e) + 2.0));
    if (r > static_cast<uint32_t>(m)) r = static_cast<uint32_t>(m);
    uint32_t unused;
    block_select<KB, 2>(KeyArraySrc{sample}, RankByKey{}, m, r, c.rhist, c, t_lo, unused);
    const uint32_t range = key_max > t_lo ? key_max - t_lo : 0u;
    const int bits = 32 - __clz(range);
    bin_shift = bits > kBinBits - 1 ? bits - (kBinBits - 1) : 0;
}

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

// Keeps the staged elements whose key is >= t_lo.  Each thread first loads
// its vectors into registers and marks passing elements in a bit mask; one
// block scan then gives every thread its output slot, so candidates are
// written without per-element atomics.  `reserve(total)` (thread 0) returns
// the first slot; `put(slot, raw, col)` stores one candidate.  The key of
// each candidate is also counted in hist (kBins bins).  Returns the number
// of candidates of the chunk (block-uniform).
template <int DT, class Reserve, class Put>
__device__ uint32_t filter_chunk(const typename Elem<DT>::raw_t *stage, int off, int64_t len,
                                 int64_t col_base, uint32_t t_lo, int bin_shift, uint32_t *hist,
                                 Ctrl &c, Reserve &&reserve, Put &&put) {
    constexpr int es = Elem<DT>::kBytes;
    constexpr int EPV = 16 / es;
    constexpr int VPT = (kChunkBytes + 16) / 16 / kThreads + 1;
    const int64_t nvec = ((off + len) * es + 15) / 16;
    const uint4 *svec = reinterpret_cast<const uint4 *>(stage);
    uint4 w[VPT];
    uint32_t msk[VPT];
    uint32_t cnt = 0;
    const float tf = __uint_as_float((t_lo & 0x80000000u) ? (t_lo & 0x7FFFFFFFu) : ~t_lo);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t v = threadIdx.x + static_cast<int64_t>(j) * kThreads;
        w[j] = v < nvec ? svec[v] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t v = threadIdx.x + static_cast<int64_t>(j) * kThreads;
        // lanes of this vector that hold elements [0, len)
        const int64_t e0 = v * EPV - off;
        int lo = e0 < 0 ? static_cast<int>(-e0) : 0;
        int hi = (len - e0) < EPV ? static_cast<int>(len - e0) : EPV;
        uint32_t valid = 0;
        if (v < nvec && hi > lo) valid = ((1u << hi) - 1u) & ~((1u << lo) - 1u);
        uint32_t m = 0;
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
            const uint32_t raw = vec_elem<es>(w[j], q);
            const bool pass = es == 4 ? __uint_as_float(raw) >= tf : Elem<DT>::key(raw) >= t_lo;
            m |= static_cast<uint32_t>(pass) << q;
        }
        msk[j] = m & valid;
        cnt += __popc(msk[j]);
    }
    uint32_t total;
    const uint32_t excl = block_excl_scan(cnt, c, total);
    if (threadIdx.x == 0) c.bcast[0] = reserve(total);
    __syncthreads();
    uint32_t slot = c.bcast[0] + excl;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        uint32_t m = msk[j];
        const int64_t v = threadIdx.x + static_cast<int64_t>(j) * kThreads;
        while (m) {
            const int q = __ffs(m) - 1;
            m &= m - 1;
            const uint32_t raw = vec_elem<es>(w[j], q);
            atomicAdd(&hist[bin_of(Elem<DT>::key(raw), t_lo, bin_shift)], 1u);
            put(slot++, raw, static_cast<uint32_t>(col_base + v * EPV + q - off));
        }
    }
    __syncthreads();
    return total;
}

// Finds the exact top-k among `total` (>= k) candidates whose keys are
// counted in hist[kBins] (shared memory): the bin b* holding the k-th key
// from the top, every candidate of a higher bin, and the best `need` of bin
// b* (ranked by key, then by smaller column).  Writes sel[0..k).  Returns
// false when bin b* holds more candidates than `bcap` (caller falls back).
// `sel` may alias `hist` (the histogram is consumed first).
template <int DT, class CandSrc>
__device__ bool select_from_candidates(const CandSrc &cands, uint32_t total, uint32_t *hist,
                                       uint32_t t_lo, int bin_shift, int k, bool det, uint2 *sel,
                                       uint2 *blist, uint32_t bcap, Ctrl &c) {
    constexpr int BPT = kBins / kThreads;
    constexpr int KB = Elem<DT>::kKeyBits;
    uint32_t local[BPT], s = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        local[j] = hist[kBins - 1 - BPT * threadIdx.x - j];
        s += local[j];
    }
    uint32_t tot;
    const uint32_t excl = block_excl_scan(s, c, tot);
    if (excl < static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= excl + s) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            if (acc + local[j] >= static_cast<uint32_t>(k)) {
                c.bcast[2] = kBins - 1 - BPT * threadIdx.x - j;
                c.bcast[3] = acc;
                c.bcast[4] = local[j];
                break;
            }
            acc += local[j];
        }
    }
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
        // rank every member of bin b* against the others: a total order by
        // (key desc, column asc); the first `need` ranks are selected
        for (uint32_t i = threadIdx.x; i < bsize; i += blockDim.x) {
            const uint2 me = blist[i];
            const uint32_t mk = Elem<DT>::key(me.x);
            uint32_t rank = 0;
            for (uint32_t j = 0; j < bsize; ++j) {
                const uint2 o = blist[j];
                const uint32_t ok = Elem<DT>::key(o.x);
                rank += (ok > mk || (ok == mk && o.y < me.y)) ? 1u : 0u;
            }
            if (rank < need) sel[above + rank] = me;
        }
        __syncthreads();
    } else {
        const PairSrc<DT> bs{blist};
        uint32_t t, gt;
        block_select<KB, KB / 8>(bs, RankByKey{}, bsize, need, c.rhist, c, t, gt);
        const uint32_t need_ties = need - gt;
        uint32_t col_max = 0xFFFFFFFFu;
        if (det) {
            uint32_t kk, g2;
            block_select<32, 4>(bs, RankTieColumn{t}, bsize, need_ties, c.rhist, c, kk, g2);
            col_max = ~kk;
        }
        collect<DT>(bs, bsize, t, gt, need_ties, det, col_max, sel, above, c);
    }
    return true;
}

// Samples m keys of a row staged in shared memory (single elements at a
// fixed stride) into `sample`, and their maximum into c.key_max.
template <int DT>
__device__ void sample_staged(const typename Elem<DT>::raw_t *row, int64_t n, int m, uint32_t *sample,
                              Ctrl &c) {
    if (threadIdx.x == 0) c.key_max = 0;
    __syncthreads();
    uint32_t kmax = 0;
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const uint32_t key = Elem<DT>::key(row[static_cast<int64_t>(i) * n / m]);
        sample[i] = key;
        kmax = key > kmax ? key : kmax;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, kmax, o);
        kmax = y > kmax ? y : kmax;
    }
    if (lane_id() == 0) atomicMax(&c.key_max, kmax);
    __syncthreads();
}

// ---------------------------------------------------------------- kernels

// Guess kernel: one block per split row computes the row's threshold guess
// from a strided sample (256 groups of 8 consecutive columns), anchored at
// the hint's argmax column when a hint is given, and stores it in the row's
// workspace header.  It lets the main kernel launch at once (programmatic
// dependent launch), so the main kernel's bulk copies overlap this work.
template <int DT>
__global__ void __launch_bounds__(kThreads) guess_kernel(const __grid_constant__ Params p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ Ctrl c;
    __shared__ uint32_t sample[kSampleSize];
    const int64_t row = blockIdx.x;
    int64_t n, col0;
    row_window(p, row, n, col0);
    if (n <= p.k || n <= p.plan.chunk) return;
    const typename Elem<DT>::raw_t *xrow =
        static_cast<const typename Elem<DT>::raw_t *>(p.x) + row * p.row_stride + col0;
    if (threadIdx.x == 0) c.key_max = 0;
    const int64_t pos = static_cast<int64_t>(threadIdx.x) * (n - 8) / (kSampleGroups - 1);
    uint32_t kmax = 0;
    uint32_t raw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) raw[j] = ldg_raw(xrow + pos + j);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t key = Elem<DT>::key(raw[j]);
        sample[threadIdx.x * 8 + j] = key;
        kmax = key > kmax ? key : kmax;
    }
    if (threadIdx.x == 0 && p.pre_idx) {  // hint anchor: previous argmax
        const int32_t a = __ldg(p.pre_idx + (row / p.next_n) * p.k);
        if (static_cast<uint64_t>(static_cast<uint32_t>(a)) < static_cast<uint64_t>(n)) {
            const uint32_t key = Elem<DT>::key(ldg_raw(xrow + a));
            kmax = key > kmax ? key : kmax;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, kmax, o);
        kmax = y > kmax ? y : kmax;
    }
    __syncthreads();
    if (lane_id() == 0) atomicMax(&c.key_max, kmax);
    __syncthreads();
    uint32_t t_lo;
    int bin_shift;
    guess_threshold<DT>(sample, kSampleSize, n, p.k, c.key_max, c, t_lo, bin_shift);
    if (threadIdx.x == 0) {
        uint32_t *rhdr = reinterpret_cast<uint32_t *>(p.ws + kWsHeaderBytes +
                                                      static_cast<size_t>(row) * p.plan.ws_row_bytes);
        rhdr[3] = t_lo;
        rhdr[4] = static_cast<uint32_t>(bin_shift);
    }
}

// Main kernel: block b handles chunk b % C of row b / C.
template <int DT>
__global__ void __launch_bounds__(kThreads) topk_kernel(const __grid_constant__ Params p) {
    using raw_t = typename Elem<DT>::raw_t;
    extern __shared__ __align__(128) uint8_t smem[];
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + p.plan.off_hist);
    uint2 *sel = reinterpret_cast<uint2 *>(smem + p.plan.off_hist);  // aliases hist
    raw_t *stage = reinterpret_cast<raw_t *>(smem + p.plan.off_stage);
    const uint32_t stage_pairs = static_cast<uint32_t>((p.plan.smem - p.plan.off_stage) / sizeof(uint2));

    const int cpr = p.plan.chunks_per_row;
    const int64_t row = static_cast<int64_t>(blockIdx.x) / cpr;
    const int chunk = static_cast<int>(blockIdx.x % cpr);
    const int k = p.k;
    const bool det = p.deterministic != 0;

    GBTOPK_TRACE_POINT(0, 0);
    int64_t n, col0;
    row_window(p, row, n, col0);
    GBTOPK_TRACE_POINT(1, 0);
    const raw_t *xrow = static_cast<const raw_t *>(p.x) + row * p.row_stride + col0;

    // ---- short and empty rows: every valid column, then -1
    if (n <= k) {
        GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | (chunk ? 0u : 1u));
        if (chunk != 0) return;
        const bool need_raw = det || p.out_val != nullptr;
        for (int j = threadIdx.x; j < n; j += blockDim.x)
            sel[j] = make_uint2(need_raw ? ldg_raw(xrow + j) : 0u, static_cast<uint32_t>(j));
        __syncthreads();
        if (det) sort_selection<DT>(sel, static_cast<int>(n));
        emit<DT>(p, row, sel, static_cast<int>(n));
        GBTOPK_TRACE_POINT(6, 0);
        return;
    }

    const int64_t CH = p.plan.chunk;
    const int64_t nch = (n + CH - 1) / CH;
    if (chunk >= nch) {
        GBTOPK_TRACE_POINT(7, static_cast<unsigned long long>(n) << 8);
        return;
    }

    if (threadIdx.x == 0) mbar_init(&c.bar);
    __syncthreads();

    // ---- single-chunk rows: everything in shared memory
    if (nch == 1) {
        int off;
        const uint32_t body = stage_row<DT>(xrow, n, stage, &c.bar, off);
        __syncthreads();
        const bool ok = wait_stage(p, c, body);
        GBTOPK_TRACE_POINT(3, 0);
        bool done = false;
        if (ok && n > kExactMax) {
            // sampled guess from the staged row, filter, exact select
            uint32_t *sample = hist;  // dead before the histogram is built
            sample_staged<DT>(stage + off, n, kSampleSize, sample, c);
            uint32_t t_lo;
            int bin_shift;
            guess_threshold<DT>(sample, kSampleSize, n, k, c.key_max, c, t_lo, bin_shift);
            for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            uint2 *lcand = reinterpret_cast<uint2 *>(stage);  // rows are in registers by then
            const uint32_t total = filter_chunk<DT>(
                stage, off, n, 0, t_lo, bin_shift, hist, c, [](uint32_t) { return 0u; },
                [&](uint32_t slot, uint32_t raw, uint32_t col) {
                    if (slot < stage_pairs) lcand[slot] = make_uint2(raw, col);
                });
            if (total >= static_cast<uint32_t>(k) && total <= stage_pairs) {
                done = select_from_candidates<DT>(PairSrc<DT>{lcand}, total, hist, t_lo, bin_shift, k,
                                                  det, sel, lcand + total, stage_pairs - total, c);
            }
            if (!done) exact_select<DT>(GlobalSrc<DT>{xrow}, n, k, det, sel, c.rhist, c);
            done = true;
        }
        if (!done) {
            if (ok) exact_select<DT>(StageSrc<DT>{stage + off}, n, k, det, sel, c.rhist, c);
            else exact_select<DT>(GlobalSrc<DT>{xrow}, n, k, det, sel, c.rhist, c);
        }
        if (det) sort_selection<DT>(sel, k);
        emit<DT>(p, row, sel, k);
        drain_stage(c, body, ok);
        GBTOPK_TRACE_POINT(6, 0);
        GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | 2u);
        return;
    }

    // ---- split rows
    const int64_t c0 = static_cast<int64_t>(chunk) * CH;
    const int64_t len = (n - c0) < CH ? (n - c0) : CH;
    int off;
    const uint32_t body = stage_row<DT>(xrow + c0, len, stage, &c.bar, off);
    uint8_t *wrow = p.ws + kWsHeaderBytes + static_cast<size_t>(row) * p.plan.ws_row_bytes;
    uint32_t *rhdr = reinterpret_cast<uint32_t *>(wrow);  // ticket, count, flags, t_lo, shift
    uint32_t *ghist = reinterpret_cast<uint32_t *>(wrow + kRowHeaderBytes);
    uint2 *gcand = reinterpret_cast<uint2 *>(wrow + kRowCounterBytes);
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
    // the guess kernel's results: wait for it (programmatic dependent launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t t_lo = __ldcg(&rhdr[3]);
    const int bin_shift = static_cast<int>(__ldcg(&rhdr[4]));
    GBTOPK_TRACE_POINT(2, 0);
    __syncthreads();
    const bool staged_ok = wait_stage(p, c, body);
    GBTOPK_TRACE_POINT(3, 0);
    const uint32_t gcap = static_cast<uint32_t>(p.plan.gcap);
    uint32_t lc = 0;
    if (staged_ok) {
        lc = filter_chunk<DT>(
            stage, off, len, c0, t_lo, bin_shift, hist, c,
            [&](uint32_t total) {
                const uint32_t gb = atomicAdd(&rhdr[1], total);
                if (gb + total > gcap) atomicOr(&rhdr[2], kRowOverflow);
                return gb;
            },
            [&](uint32_t slot, uint32_t raw, uint32_t col) {
                if (slot < gcap) gcand[slot] = make_uint2(raw, col);
            });
        for (int b = threadIdx.x; b < kBins; b += blockDim.x)
            if (hist[b]) atomicAdd(&ghist[b], hist[b]);
    } else if (threadIdx.x == 0) {
        atomicOr(&rhdr[2], kRowOverflow);
    }
    GBTOPK_TRACE_POINT(4, 0);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t ticket = atomicAdd(&rhdr[0], 1u);
        c.bcast[1] = (ticket == static_cast<uint32_t>(nch - 1)) ? 1u : 0u;
    }
    __syncthreads();
    GBTOPK_TRACE_POINT(5, 0);
    if (c.bcast[1] == 0u) {
        drain_stage(c, body, staged_ok);
        GBTOPK_TRACE_POINT(6, 0);
        GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | 3u);
        return;
    }

    // ---- last block of the row: exact k-th from histogram + candidates
    __threadfence();
    const uint32_t total = __ldcg(&rhdr[1]);
    const uint32_t flags = __ldcg(&rhdr[2]);
    bool fallback = flags != 0u || total < static_cast<uint32_t>(k);
    if (!fallback) {
        for (int b = threadIdx.x; b < kBins; b += blockDim.x) hist[b] = __ldcg(&ghist[b]);
        __syncthreads();
        fallback = !select_from_candidates<DT>(GlobalPairSrc<DT>{gcand}, total, hist, t_lo, bin_shift,
                                               k, det, sel, reinterpret_cast<uint2 *>(stage),
                                               stage_pairs, c);
    }
    if (fallback) exact_select<DT>(GlobalSrc<DT>{xrow}, n, k, det, sel, c.rhist, c);

    // Leave the row's counters and histogram zero-filled for the next call.
    for (int b = threadIdx.x; b < kBins; b += blockDim.x) ghist[b] = 0u;
    if (threadIdx.x < kRowHeaderBytes / 4) rhdr[threadIdx.x] = 0u;
    if (det) sort_selection<DT>(sel, k);
    emit<DT>(p, row, sel, k);
    drain_stage(c, body, staged_ok);
    GBTOPK_TRACE_POINT(6, 0);
    GBTOPK_TRACE_POINT(7, (static_cast<unsigned long long>(n) << 8) | (fallback ? 5u : 4u) |
                              (static_cast<unsigned long long>(total) << 40));
}

template <int DT>
cudaError_t launch_dt(const Params &p, cudaStream_t stream) {
    static size_t configured = 0;  // largest dynamic smem opted in so far
    if (p.plan.smem > 48 * 1024 && p.plan.smem > configured) {
        const cudaError_t e = cudaFuncSetAttribute(
            topk_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.plan.smem));
        if (e != cudaSuccess) return e;
        configured = p.plan.smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.plan.grid));
    cfg.blockDim = dim3(p.plan.threads);
    cfg.dynamicSmemBytes = p.plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.plan.split) {
        guess_kernel<DT><<<static_cast<unsigned>(p.num_rows), kThreads, 0, stream>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, topk_kernel<DT>, p);
    if (e != cudaSuccess) return e;
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

// gbtopk_varlen_static_ws: the same top-K call as gbtopk_varlen, for callers
// that cannot hand the library a device workspace.
//
// Some callers have no way to allocate device memory at the point where
// they need top-K: code that runs while a CUDA graph is being captured
// (cudaMalloc is not a capturable operation), engines whose device memory is
// owned entirely by an external allocator or memory planner that forbids
// side allocations, and plugin hosts that only pass in tensors they
// allocated themselves.  For them the scratch lives in one fixed buffer
// compiled into this module instead: kStaticWsBytes bytes of device memory
// per GPU, reserved when the module is loaded and held until the process
// exits.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "gbtopk.h"

namespace {

// 16 MiB: enough for, e.g., a 64 x 163840 fp32 decode batch with top_k 2048
// (about 6.3 MiB); larger geometries are refused.
constexpr size_t kStaticWsBytes = size_t{16} << 20;
constexpr int kMaxDevices = 64;

// Scratch shared by every call on a device.  Its contents carry over from
// one call to the next; the kernels write every scratch byte they read
// within a call, so nothing has to be cleared between calls (the first four
// bytes collect device status flags, and start at zero).
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

std::mutex g_mutex;
void *g_dev_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, looked up once per
// device (the host-side symbol is only a handle; the kernels need the
// address the runtime assigned on that device).  The cached address belongs
// to the device's current context: after cudaDeviceReset it is stale, so
// this entry point must not be used again in that process.
int static_ws_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return GBTOPK_ECUDA;
    if (dev >= kMaxDevices) return GBTOPK_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_dev_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) return GBTOPK_ECUDA;
        g_dev_ptr[dev] = ptr;
    }
    *out = g_dev_ptr[dev];
    return GBTOPK_OK;
}

}  // namespace

extern "C" {

int gbtopk_varlen_static_ws(const void *logits, int dtype, int64_t num_rows, int64_t width,
                            int64_t row_stride, const int32_t *seq_lens, int32_t next_n,
                            int32_t compress_ratio, int32_t top_k, const int32_t *pre_idx,
                            int32_t *out_indices, void *out_values, int deterministic,
                            void *stream) {
    // Refuse, before touching the device, a geometry the library does not
    // plan (with gbtopk_varlen's own status) or whose scratch does not fit
    // in the built-in buffer.
    int64_t plan[13];
    const int prc = gbtopk_plan_query(num_rows, width, top_k, dtype, plan);
    if (prc != GBTOPK_OK) return prc;
    if (static_cast<size_t>(plan[8]) > kStaticWsBytes) return GBTOPK_EWORKSPACE;
    void *ws = nullptr;
    const int rc = static_ws_address(&ws);
    if (rc != GBTOPK_OK) return rc;
    return gbtopk_varlen(logits, dtype, num_rows, width, row_stride, seq_lens, next_n,
                         compress_ratio, top_k, pre_idx, out_indices, out_values, deterministic,
                         ws, kStaticWsBytes, stream);
}

}  // extern "C"

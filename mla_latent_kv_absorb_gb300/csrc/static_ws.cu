// static_ws.cu -- mla_decode_paged_static_ws: the paged decode plus the split merge with the
// split-partial scratch held in a fixed device array of this library, so that the call itself
// allocates nothing (declared in include/mla.h).
//
// Who needs it: callers that cannot allocate device memory at the point of the call -- code
// running inside a custom allocator's own callbacks, runtimes that pre-reserve all device memory
// and forbid later allocation, or embedders without a caching allocator of their own.  The
// regular entry points take the workspace from the caller; this one takes it from the array below.
//
// The array lives in its own translation unit, hence in its own module: its storage is reserved
// when that module is loaded.  Under the CUDA runtime's default lazy module loading that is the
// first call on each device, and code that never calls this entry point never pays for it; with
// CUDA_MODULE_LOADING=EAGER every device that creates a context loads the module, and holds the
// array, from the start.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/mla.h"

namespace mla {
void set_last_error_text(const char* text);
}

namespace {

constexpr size_t kPartialBytes = (size_t)128 * 512 * sizeof(float) + (size_t)128 * sizeof(float);
static_assert(MLA_STATIC_WS_BYTES == (size_t)MLA_STATIC_WS_MAX_PARTIALS * kPartialBytes,
              "static workspace size must match the partial layout");

// Split partials of one call: [num_partials][128][512] fp32 then [num_partials][128] fp32.
// Nothing in it needs to start at zero: the decode launch of a call writes every partial that
// the merge launch of the same call reads.
static __device__ __align__(256) float g_static_ws[MLA_STATIC_WS_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_ws_ptr[kMaxDevices] = {};

// Address of g_static_ws on the current device, looked up once per device and kept for the life
// of the process: valid only while the device's primary context lives (a cudaDeviceReset would
// reload the module, perhaps elsewhere; the header tells callers not to use this entry point
// after one).
mla_status static_ws_ptr(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        char msg[160];
        snprintf(msg, sizeof msg, "cudaGetDevice: %s (device %d, at most %d supported)",
                 e == cudaSuccess ? "ok" : cudaGetErrorString(e), dev, kMaxDevices);
        mla::set_last_error_text(msg);
        return MLA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_ws_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p) {
            char msg[200];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static workspace) on device %d: %s (%s)", dev,
                     cudaGetErrorString(e), cudaGetErrorName(e));
            mla::set_last_error_text(msg);
            return MLA_ERR_CUDA;
        }
        g_ws_ptr[dev] = p;
    }
    *out = g_ws_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_paged_static_ws(const mla_plan_info* info, const void* plan_dev, const void* q_abs,
                                                 const void* q_r, mla_kv_dtype kv_dtype, const void* kv_pool,
                                                 const float* kv_scale, const void* kr_pool, int32_t num_pool_pages,
                                                 const int32_t* block_table, int32_t max_pages_per_seq,
                                                 float softmax_scale, void* o_lat, float* lse, uint32_t* dev_error,
                                                 void* stream)
{
    if (!info) return MLA_ERR_INVALID_ARG;
    if (info->num_partials < 0 || info->num_partials > MLA_STATIC_WS_MAX_PARTIALS ||
        info->workspace_bytes > (int64_t)MLA_STATIC_WS_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "plan has %d split partials (%lld bytes); the static workspace holds at most %d (%zu bytes): "
                 "plan with fewer clusters or call mla_decode_paged with a workspace",
                 info->num_partials, (long long)info->workspace_bytes, MLA_STATIC_WS_MAX_PARTIALS,
                 (size_t)MLA_STATIC_WS_BYTES);
        mla::set_last_error_text(msg);
        return MLA_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    if (info->workspace_bytes > 0) {
        const mla_status st = static_ws_ptr(&ws);
        if (st != MLA_OK) return st;
    }
    const size_t ws_bytes = ws ? (size_t)MLA_STATIC_WS_BYTES : 0;
    mla_status st = mla_decode_paged(info, plan_dev, q_abs, q_r, kv_dtype, kv_pool, kv_scale, kr_pool, num_pool_pages,
                                     block_table, max_pages_per_seq, softmax_scale, ws, ws_bytes, o_lat, lse,
                                     dev_error, stream);
    if (st != MLA_OK) return st;
    return mla_combine_splits(info, plan_dev, ws, ws_bytes, o_lat, lse, stream);
}

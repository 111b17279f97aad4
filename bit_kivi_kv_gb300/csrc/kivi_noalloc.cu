// Decode attention for callers that cannot allocate device memory.
//
// kivi_decode_attn needs a device workspace for the split-KV partial results,
// and the caller provides it.  Some callers cannot: a plugin running inside a
// host framework that owns all device memory through its own pool (where a
// raw cudaMalloc is refused, or would synchronize the device and stall the
// framework's other streams), or code that is only ever handed device
// pointers and has no allocator of its own.  For them this file keeps one
// workspace in a file-scope device array and runs the same decode path on it.
#include <stdio.h>

#include <mutex>

#include "kivi_common.cuh"

namespace {

constexpr size_t kStaticWorkspaceBytes = (size_t)16 << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device

}  // namespace

// The workspace itself.  Every device that loads this code holds it until the
// process exits.  Host code must not pass this name to a kernel: on the host it
// is only a stand-in symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char kivi_static_decode_workspace[kStaticWorkspaceBytes];

extern "C" kivi_status kivi_decode_attn_static_ws(kivi_cache_t cache, const void* q, void* out,
                                                  float softmax_scale, kivi_stream_t stream) {
    char msg[256];
    if (!cache) return kivi::report_error(KIVI_ERR_INVALID_ARG, "null handle");
    const size_t need = kivi::decode_workspace_need(cache);
    if (need > kStaticWorkspaceBytes) {
        snprintf(msg, sizeof msg,
                 "this cache shape needs %zu bytes of decode workspace, more than the %zu-byte static "
                 "workspace; use kivi_decode_attn with a caller-provided workspace",
                 need, kStaticWorkspaceBytes);
        return kivi::report_error(KIVI_ERR_CAPACITY, msg);
    }
    // the workspace must be the cache's device's array: that device must be current
    const kivi_status sdev = kivi::cache_device(cache);
    if (sdev != KIVI_OK) return sdev;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
        return kivi::report_error(KIVI_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) return kivi::report_error(KIVI_ERR_UNSUPPORTED, "device index too large");
    void* ws = nullptr;
    {
        // First call on this device (with it current): look up the array's
        // address.  The library's modules load lazily, so this lookup is also
        // what loads the array onto the device and reserves its bytes there.
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        ws = g_scratch_addr[dev];
        if (!ws) {
            e = cudaGetSymbolAddress(&ws, kivi_static_decode_workspace);
            if (e != cudaSuccess || !ws) {
                snprintf(msg, sizeof msg,
                         "could not load the %zu-byte static decode workspace on device %d "
                         "(cudaGetSymbolAddress: %s)",
                         kStaticWorkspaceBytes, dev, cudaGetErrorString(e));
                return kivi::report_error(KIVI_ERR_CUDA, msg);
            }
            g_scratch_addr[dev] = ws;
        }
    }
    // Nothing in the workspace needs to start at zero: each call writes every
    // partial result before the merge reads it.
    return kivi_decode_attn(cache, q, out, softmax_scale, ws, kStaticWorkspaceBytes, stream);
}

// conv2d_fwd for callers that must not allocate device memory.
//
// Who needs it: code that runs where a cudaMalloc is not allowed or not
// affordable — inference plugins whose host application owns every byte of
// device memory and hands out only input/output buffers, real-time loops that
// cannot take the device-wide synchronisation a cudaMalloc/cudaFree may
// cause, and processes that run under a fixed memory cap set by someone
// else.  Such a caller cannot provide the workspace conv2d_fwd asks for.
//
// This file gives them one entry point, conv2d_fwd_static_workspace, whose
// scratch lives in a file-scope __device__ array of fixed size.  The array is
// part of the library's device image: every GPU that loads the library holds
// it until the process exits.  Host code cannot use the array's name as a
// device address (on the host it names a stand-in object), so the device
// address is looked up once per device with cudaGetSymbolAddress, on the
// first call made while that device is current, and cached for the life of
// the process (valid while the device's primary context is not reset).
#include <mutex>

#include "internal.h"

#define CONV2D_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kStaticWorkspaceBytes = CONV2D_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_lock;
void* g_device_addr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device (set-up on the
// first call per device).  Returns CONV2D_ERR_CUDA when the lookup fails.
conv2d_status static_workspace_addr(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CONV2D_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_device_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return CONV2D_ERR_CUDA;
        g_device_addr[dev] = p;
    }
    *out = g_device_addr[dev];
    return CONV2D_OK;
}

}  // namespace

CONV2D_API conv2d_status conv2d_fwd_static_workspace(conv2d_desc_t d, const void* x, const void* w, void* y,
                                                     void* stream) {
    if (!d) return CONV2D_ERR_NULL_PTR;
    size_t need = 0;
    conv2d_status st = conv2d_workspace_size(d, &need);
    if (st != CONV2D_OK) return st;
    if (need > kStaticWorkspaceBytes) return CONV2D_ERR_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    if (need > 0) {
        st = static_workspace_addr(&ws);
        if (st != CONV2D_OK) return st;
    }
    // Every byte the kernels read from the workspace is written earlier in the
    // same call, so leftovers from a previous call need no clearing.
    return conv2d_fwd(d, x, w, y, ws, need > 0 ? kStaticWorkspaceBytes : 0, stream);
}

CONV2D_API conv2d_status conv2d_static_workspace_bytes(size_t* bytes) {
    if (!bytes) return CONV2D_ERR_NULL_PTR;
    *bytes = kStaticWorkspaceBytes;
    return CONV2D_OK;
}

// noalloc.cu -- gdr_bwd_run_noalloc: the whole backward without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need the backward: a plugin
// that runs inside another framework and may only touch the tensors it is handed, a service with a
// fixed device-memory budget that forbids allocations after start-up, or a latency-sensitive loop in
// which cudaMalloc's implicit device synchronisation is not acceptable.  For them the scratch memory
// lives in a file-scope __device__ array of GDR_BWD_NOALLOC_MAX_WORKSPACE bytes.  Every GPU that loads
// this library holds that array until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it names a stand-in object),
// so the first call on each device looks the address up with cudaGetSymbolAddress while that device is
// current, and caches it per device.  That first call should therefore happen before any stream
// capture begins.  All calls share the one array and it keeps whatever the last call left: the
// backward clears what must start at zero (its status word) and overwrites everything else before
// reading it, and calls that overlap on the GPU race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdr_bwd.h"

namespace {

constexpr size_t kScratchBytes = GDR_BWD_NOALLOC_MAX_WORKSPACE;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
gdr_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GDR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDR_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDR_OK;
}

}  // namespace

// The status word of the last run_noalloc on the current device lives in the shared array, where
// gdr_bwd_get_status finds it given the array's address as the workspace.
extern "C" gdr_status gdr_bwd_get_status_noalloc(gdr_bwd_plan *plan, void *stream) {
    if (!plan) return GDR_ERR_INVALID_ARG;
    if (gdr_bwd_workspace_bytes(plan) > kScratchBytes) return GDR_ERR_UNSUPPORTED;
    void *ws = nullptr;
    gdr_status st = scratch_address(&ws);
    if (st != GDR_OK) return st;
    return gdr_bwd_get_status(plan, ws, stream);
}

extern "C" gdr_status gdr_bwd_run_noalloc(gdr_bwd_plan *plan, const gdr_bwd_args *args, void *stream) {
    if (!plan || !args) return GDR_ERR_INVALID_ARG;
    if (gdr_bwd_workspace_bytes(plan) > kScratchBytes) return GDR_ERR_UNSUPPORTED;
    void *ws = nullptr;
    gdr_status st = scratch_address(&ws);
    if (st != GDR_OK) return st;
    return gdr_bwd_run(plan, args, ws, kScratchBytes, stream);
}

// gdn_noalloc.cu -- gdn_segmented_fwd for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework that owns all device memory through
// its own pool and forbids side allocations, a request path that must not take the implicit
// synchronisation and latency of an allocation, or a program that only holds buffers it
// imported from another process. They can still pass their inputs and outputs; this entry
// point supplies the segmented forward's scratch (segment summaries, scanned states, the
// device error word) from one fixed array in the library's own device memory instead of a
// caller workspace.
//
// The array is a file-scope __device__ variable of GDN_NOALLOC_SCRATCH_BYTES bytes: every GPU
// that loads this library holds it until the process exits. Host code cannot use the
// array's name as a device address, so the first call on each device looks its address up
// with cudaGetSymbolAddress (with that device current) and caches it. The cache is keyed by
// device number, which assumes the runtime's primary context: with another driver context
// current, or after cudaDeviceReset, the cached address would belong to a context that is
// gone, so those uses are documented as unsupported.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void* g_scratch_addr[kMaxDevices] = {};

// Address of this device's copy of the array; nullptr if the lookup failed.
void* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> guard(g_setup_lock);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" gdn_status gdn_segmented_fwd_noalloc(const gdn_problem* p, int nseg, const void* q,
                                                const void* k, const void* v, const void* g,
                                                const void* beta, const float* h0, void* o,
                                                float* h_final, unsigned* device_error,
                                                void* stream) {
    const size_t need = gdn_workspace_bytes(p, nseg);
    if (need == 0) {
        // invalid problem: let the regular entry point name the reason (it launches nothing)
        return gdn_segmented_fwd(p, nseg, q, k, v, g, beta, h0, o, h_final, nullptr, nullptr,
                                 0, stream);
    }
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    if (device_error && (reinterpret_cast<uintptr_t>(device_error) & 7u)) return GDN_ERR_MISALIGNED;
    void* scratch = scratch_for_current_device();
    if (!scratch) return GDN_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the error word must start at zero
    if (cudaMemsetAsync(scratch, 0, sizeof(gdn::DeviceError), s) != cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_status st = gdn_segmented_fwd(p, nseg, q, k, v, g, beta, h0, o, h_final, nullptr,
                                      scratch, (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
    if (st != GDN_OK) return st;
    if (device_error &&
        cudaMemcpyAsync(device_error, scratch, sizeof(gdn::DeviceError), cudaMemcpyDeviceToDevice,
                        s) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

// noalloc.cu -- a fixed block of device memory for callers that must not allocate.
//
// Some callers cannot let this library call cudaMalloc: code embedded in a
// host application that owns every device allocation and forbids others,
// real-time loops that cannot absorb the implicit synchronisation an
// allocation may cause, and programs that have already handed all free
// device memory to their own allocator.  For them,
// tropical_permute_trace_noalloc keeps the partial results of a split
// reduction in the array below instead of pool workspace.
//
// The array lives in the module for as long as the library is loaded, on
// every GPU that loads it.  Its name is only a host-side stand-in in host
// code: kernels must be given the device address that cudaGetSymbolAddress
// returns, looked up here once per device with that device current and kept
// for the life of the process (like the rest of the library's per-device
// state, it does not survive a cudaDeviceReset).
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace trop {

// 256 KiB: 21845 partial results of f32/i32 (12 bytes each) or 16384 of f64/i64 (16 bytes);
// a split reduction makes fewer than 16 x (SM count) of them
constexpr size_t NOALLOC_SCRATCH_BYTES = 256 * 1024;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

int noalloc_scratch(void** ptr, size_t* bytes)
{
    static std::mutex mu;
    static void* addr[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(TROP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return cuda_error(e, "cudaGetSymbolAddress (fixed scratch)");
        addr[dev] = p;
    }
    *ptr = addr[dev];
    *bytes = NOALLOC_SCRATCH_BYTES;
    return TROP_OK;
}

}  // namespace trop

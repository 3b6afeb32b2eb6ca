// lrkv_decode_noalloc: lrkv_decode for callers that cannot allocate device
// memory.  The decode's scratch (launch plan, private queries and per-segment
// partial softmax states) lives in one file-scope device array that is part
// of the library image, so the caller passes only inputs and outputs.
#include <mutex>

#include "decode_kernels.cuh"

namespace lrkv {

// Device-resident scratch shared by every lrkv_decode_noalloc call on a GPU.
// In host code `g_noalloc_scratch` names a host-side stand-in, not a device
// address: its device address is obtained with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LRKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).  Returns nullptr on failure.
void *noalloc_scratch_address(cudaError_t *err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_addr[dev] = p;
    }
    *err = cudaSuccess;
    return g_addr[dev];
}

}  // namespace lrkv
